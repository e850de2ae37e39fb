"""Throughput of the speculative-pipeline-decoding step (default: 4B shape, n = 8, forced p = 0.6).

One bench "step" is one pipeline step: every occupied stage runs its layers on its own
token, the draft module runs on the second stream, then the LM head and device-side
verification / rollback.  The timed region is K consecutive steps of a generation after
the (untimed) prefill; value = committed tokens / device time.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
                    [--mode forced-0.6 | greedy | t1] [--shape 4b | 8b] [--n N] [--speculate input|output]

Modes: forced-<p> (drafts equal the greedy token with probability p), greedy (the draft
module's argmax), t1 (the T = 1 workload: 4B shape, prompt 256, rejection sampling).
Shapes: tiny (fp32, L4 d256), 06b (L28 d1024, n 4), 4b (L36 d2560, prompt 512) and 8b (L36
d4096, prompt 4096, Ls 2).

Multi-GPU: independent replicas (one sequence per GPU, no collective on the data path);
value = all ranks' committed tokens / max-over-ranks time.
"""
from __future__ import annotations

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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import spd_inputs as si  # noqa: E402

METRIC = "committed tokens/s + step us (4B-shape bf16, n=8); weight GB/s vs 8 TB/s HBM"
WL = si.SHAPE_4B
NOMINAL_HBM_GBS = 8000.0     # the metric's stated HBM peak


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=16)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--mode", default="forced-0.6", help="forced-<p>, greedy (draft-module argmax) or t1 (T = 1)")
    ap.add_argument("--shape", default="4b", choices=["tiny", "06b", "4b", "8b"])
    ap.add_argument("--n", type=int, default=0, help="pipeline stages (default: the workload's)")
    ap.add_argument("--speculate", default="input", choices=["input", "output"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--skip-e2e", action="store_true", help="profiling runs: leave out the host-buffer leg")
    ap.add_argument("--layers", type=int, default=0,
                    help="profiling runs only: a smaller case of the same kernels (L layers, anchors scaled)")
    return ap.parse_args()


def mode_p(mode: str):
    return float(mode.split("-", 1)[1]) if mode.startswith("forced-") else None


def mode_temperature(mode: str) -> float:
    return 1.0 if mode == "t1" else 0.0


def alpha_ref(mode: str, n: int):
    """The commit rate both CPU figures convert steps/s with: the closed form for forced
    drafts (renewal argument: 1 / (1 + (n - 1)(1 - p))), 1/n for greedy drafting by the
    random-init draft module (its argmax never matches the target's, so every commit
    takes the n steps of a refill), None at T = 1 (no closed form)."""
    p = mode_p(mode)
    if p is not None:
        return 1.0 if p >= 1.0 else 1.0 / (1.0 + (n - 1) * (1.0 - p))
    if mode == "greedy":
        return 1.0 / n
    return None


def select_workload(args) -> si.Workload:
    """The bench workload: shape and mode select one of the workloads' model sizes."""
    if args.mode == "t1":
        wl = si.SHAPE_4B_T1
    else:
        wl = {"tiny": si.TINY, "06b": si.SHAPE_06B, "4b": si.SHAPE_4B, "8b": si.SHAPE_8B}[args.shape]
    if args.n:
        wl = si.Workload(wl.name, wl.dims, n=args.n, anchors=wl.anchors, Ls=wl.Ls, prompt_len=wl.prompt_len,
                         max_new=wl.max_new, temperature=wl.temperature, forced_p=wl.forced_p)
    return wl


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except OSError:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}, "fallback"


def dist_setup(args):
    """One process per GPU (torchrun's env).  The ranks are replicas: each decodes its own
    sequence, and the only collectives are the barrier around the timed region and the two
    scalar reductions of the result.  SPD_DIST_BACKEND=gloo runs the same code on CPU."""
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        backend = os.environ.get("SPD_DIST_BACKEND", "nccl")
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def allreduce(x: float, op, ws):
    if ws == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=op)
    return float(t.item())


L2_BYTES = 129e6   # GB300 L2


def l2_note(bytes_per_step: float) -> str:
    """How the timed steps relate to the L2: the weights streamed per step against its size
    (no flush between steps when they exceed it many times over)."""
    if bytes_per_step > 8 * L2_BYTES:
        return f"no flush needed: {bytes_per_step / 1e9:.2f} GB of weights streamed per step >> 129 MB L2"
    return (f"L2-resident: {bytes_per_step / 1e6:.0f} MB of weights per step fit the 129 MB L2 (a parity "
            "workload, not a roofline one); not flushed")


def job_value(ms_max: float, commits_all: float) -> float:
    """Whole-job committed tokens/s: every rank's commits over the slowest rank's time."""
    return commits_all / (ms_max / 1e3)


class Clocks:
    """nvidia-smi sampler running during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", str(index), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                                       "-lms", "100"], stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.p = None

    def stop(self):
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.p.terminate()
        self.p.wait()
        self.f.seek(0)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.f:
            c = [x.strip() for x in line.split(",")]
            if len(c) < 9:
                continue
            try:
                sm.append(float(c[1]))
                mx = float(c[2])
            except ValueError:
                continue
            for nm, v in zip(names, c[5:9]):
                if v.lower() in ("active", "0x1") or v == "1":
                    reasons.add(nm)
        os.unlink(self.f.name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def source_hash(path):
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def stage_sizes(L, n):
    b = [(s * L) // n for s in range(n + 1)]
    return [b[s + 1] - b[s] for s in range(n)]


def gateup_bytes(trace, dm, n):
    """Algorithmic bytes of every gate/up launch in the traced steps: per launch (round j)
    the occupied stages that hold a j-th layer stream 2 x F x d bf16 weights."""
    sizes = stage_sizes(dm.L, n)
    J = max(sizes)
    per = 2 * dm.F * dm.d * (2 if dm.dtype == "bf16" else 4)
    tot, launches = 0, 0
    for r in trace:
        m = r["n_active"]
        for j in range(J):
            tot += per * sum(1 for s in range(m) if j < sizes[s])
            launches += 1
    return tot, launches


# ---------------------------------------------------------------------------------------
def run_gb300(args, ws, rank, local):
    from speculative_pipeline_decoding_spd_gb300.engine import Engine
    dm, n = WL.dims, WL.n
    p = mode_p(args.mode)
    with si.on_device("cuda"):
        tg = si.make_target(dm, 0)
        pd = si.make_pdm(dm, WL.Ls, len(WL.anchors), 0)
    prompt = torch.from_numpy(si.make_prompt(dm.V, WL.prompt_len, 1 + rank)).cuda()
    T = mode_temperature(args.mode)
    spec = dict(speculate=args.speculate, temperature=T)
    # the generation must outlast warmup + timed steps
    alpha_lo = 1.0 / n if p is None else 1.0 / (1.0 + (n - 1) * (1.0 - p))
    if T > 0:
        alpha_lo = 1.0     # sampled drafts are often kept: size for one commit per step
    max_new = max(WL.max_new, int(math.ceil((args.warmup + args.steps + 2 * n) * min(1.0, alpha_lo * 1.3))) + 8)
    max_seq = WL.prompt_len + max_new + n + 8
    forced_ref = None
    if p is not None:
        # forced drafts follow this implementation's own greedy stream (one stage = plain decode)
        ar = Engine(dm, tg, pd, 1, WL.anchors, max_seq=max_seq, max_new=max_new + n + 2, graph=True)
        out, cnt, _ = ar.generate(prompt)
        forced_ref = torch.cat([prompt, out[:cnt], torch.zeros(n + 8, dtype=torch.int32, device="cuda")]).contiguous()
        ar.close()
    # headline: the step graphs hold no timing events (events between kernels would cut the
    # programmatic launch overlap of the kernels around them)
    e = Engine(dm, tg, pd, n, WL.anchors, max_seq=max_seq, max_new=max_new, seed=2,
               force_p=(-1.0 if p is None else p), forced_ref=forced_ref, graph=True, timing=False, **spec)
    # the prefill is not part of the metric; its time is reported beside it (second of two runs)
    e.prefill(prompt)
    pf0, pf1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    pf0.record()
    e.prefill(prompt)
    pf1.record()
    torch.cuda.synchronize()
    prefill_ms = pf0.elapsed_time(pf1)
    e.step(args.warmup)
    N0 = e.stats()["N"]
    K0 = e.stats()["K"]
    torch.cuda.synchronize()
    barrier(ws)
    clk = Clocks(local)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.cudart().cudaProfilerStart()   # ncu --profile-from-start off captures only the timed region
    ev0.record()
    left = args.steps
    while left > 0:
        k = min(8, left)
        e.step(k)
        left -= k
    ev1.record()
    torch.cuda.synchronize()
    torch.cuda.cudart().cudaProfilerStop()
    clocks = clk.stop()
    barrier(ws)
    ms = ev0.elapsed_time(ev1)
    st = e.stats()
    N1, K1 = st["N"], st["K"]
    assert K1 - K0 == args.steps, "generation ended inside the timed region"
    tr = e.trace()[K0:K1]
    commits = N1 - N0
    # weight bytes streamed by the timed steps (occupied stages + draft module + LM head)
    sizes = stage_sizes(dm.L, n)
    el = 2 if dm.dtype == "bf16" else 4
    layer_b = el * ((dm.Hq + 2 * dm.Hkv) * dm.hd * dm.d + dm.d * dm.Hq * dm.hd + 3 * dm.F * dm.d)
    pdm_b = el * (dm.d * len(WL.anchors) * dm.d) + WL.Ls * layer_b
    lm_b = el * dm.V * dm.d
    wbytes = sum(layer_b * sum(sizes[s] for s in range(r["n_active"])) for r in tr) + len(tr) * (pdm_b + lm_b)
    e.close()
    del e

    # roofline kernel: a second timed region of the same workload whose step graphs record a
    # CUDA event pair around every gate/up launch on its stream (spd_kernel_timing)
    er = Engine(dm, tg, pd, n, WL.anchors, max_seq=max_seq, max_new=max_new, seed=2,
                force_p=(-1.0 if p is None else p), forced_ref=forced_ref, graph=True, timing=True, **spec)
    er.prefill(prompt)
    er.step(args.warmup)
    t0_ms, l0 = er.kernel_timing()
    Kr0 = er.stats()["K"]
    left = args.steps
    while left > 0:
        k = min(8, left)
        er.step(k)
        left -= k
    torch.cuda.synchronize()
    t1_ms, l1 = er.kernel_timing()
    trr = er.trace()[Kr0:er.stats()["K"]]
    gb, gl = gateup_bytes(trr, dm, n)
    g_ms = t1_ms - t0_ms
    assert l1 - l0 == gl, (l1 - l0, gl)
    er.close()
    del er

    # ---- end to end through the public call with host buffers (prefill included)
    if args.skip_e2e:
        return dict(ms=ms, commits=commits, steps=args.steps, wbytes=wbytes, gate_bytes=gb, gate_ms=g_ms,
                    gate_launches=gl, clocks=clocks, alpha=commits / args.steps, e2e_tokens=0, e2e_s=float("nan"),
                    prefill_ms=prefill_ms,
                    e2e_steps=1, max_new=max_new, prompt_len=WL.prompt_len,
                    launches_per_step=5 * max(sizes) + 1 + 5 * WL.Ls + 2)
    e2 = Engine(dm, tg, pd, n, WL.anchors, max_seq=WL.prompt_len + WL.max_new + n + 8, max_new=WL.max_new, seed=2,
                force_p=(-1.0 if p is None else p), forced_ref=forced_ref, graph=True, **spec)
    host_prompt = prompt.cpu().numpy()
    e2.generate(host_prompt, on_host=True)   # warm
    torch.cuda.synchronize()
    t = time.perf_counter()
    toks, st2 = e2.generate(host_prompt, on_host=True)
    e2_s = time.perf_counter() - t
    e2_steps = st2.K
    e2.close()
    return dict(ms=ms, commits=commits, steps=args.steps, wbytes=wbytes, gate_bytes=gb, gate_ms=g_ms, gate_launches=gl,
                clocks=clocks, alpha=commits / args.steps, e2e_tokens=len(toks), e2e_s=e2_s, e2e_steps=e2_steps,
                prefill_ms=prefill_ms, max_new=max_new, prompt_len=WL.prompt_len,
                launches_per_step=5 * max(sizes) + 1 + 5 * WL.Ls + 2)


# ---------------------------------------------------------------------------------------
def oracle_sample(n_steps: int, mode: str, prompt_len: int = 32, e2e: bool = False):
    """The CPU oracle on the bench workload's shape: fp64 model, a short prompt (prefill
    untimed) then n_steps pipeline steps timed on all host cores.  With e2e, the workload's
    own prompt instead, and the prefill timed too.  Returns (steps/s, commits, decode s,
    prefill s, cores)."""
    from oracle import Model, SPDOracle, ar_decode
    dm = WL.dims
    tg = si.make_target(dm, 0)
    pd = si.make_pdm(dm, WL.Ls, len(WL.anchors), 0)
    m = Model(dm, tg, pd, WL.anchors)
    del tg, pd
    plen = WL.prompt_len if e2e else prompt_len
    prompt = si.make_prompt(dm.V, plen, 1)
    p = mode_p(mode)
    kw = {}
    if p is not None:
        # forced drafts follow the oracle's own greedy stream (not timed)
        ar = ar_decode(m, prompt, n_steps + 2, plen + n_steps + WL.n + 8)
        kw = dict(forced_p=p, forced_ref=list(prompt) + ar + [0] * (n_steps + WL.n + 8))
    o = SPDOracle(m, WL.n, plen + n_steps + WL.n + 8, temperature=mode_temperature(mode), seed=2, **kw)
    t = time.perf_counter()
    o.prefill(prompt)
    t_pf = time.perf_counter() - t
    t = time.perf_counter()
    for _ in range(n_steps):
        o.step()
    dt = time.perf_counter() - t
    return n_steps / dt, o.N, dt, t_pf, os.cpu_count()


def cpu_alpha(mode: str, n: int, measured: float) -> float:
    """alpha_ref where a closed form exists, else the commit rate the run measured."""
    a = alpha_ref(mode, n)
    return measured if a is None else a


def main():
    args = parse()
    global WL
    WL = select_workload(args)
    if args.layers:
        L = args.layers
        WL = si.Workload(f"{WL.name}-L{L}", si.shrink(WL.dims, L=L), n=min(WL.n, L),
                         anchors=tuple(sorted({round(a * L / 36) for a in WL.anchors})), Ls=min(WL.Ls, max(1, L // WL.n)),
                         prompt_len=WL.prompt_len, max_new=WL.max_new)
    ws, rank, local = dist_setup(args)
    if args.impl == "reference":
        return main_reference(args, ws, rank)
    torch.cuda.set_device(local)
    pk, pk_kind = peaks()
    r = run_gb300(args, ws, rank, local)
    ms_max = allreduce(r["ms"], _max_op(), ws)
    commits_all = allreduce(float(r["commits"]), _sum_op(), ws)
    if rank != 0:
        return
    p = mode_p(args.mode)
    value = job_value(ms_max, commits_all)
    hbm = pk["hbm_gbs"]
    g_ach = r["gate_bytes"] / (r["gate_ms"] / 1e3) / 1e9
    traffic = None
    tp = os.path.join(ROOT, "profiles", "gateup_traffic.json")
    if os.path.exists(tp):
        tj = json.load(open(tp))
        src = os.path.join(ROOT, "speculative_pipeline_decoding_spd_gb300", "csrc", "k_target.cu")
        if tj.get("k_target_sha") == source_hash(src) and tj.get("d") == WL.dims.d and tj.get("F") == WL.dims.F:
            per_stage_layer = tj["dram_bytes_per_stage_layer"]
            traffic = per_stage_layer * (r["gate_bytes"] / (2 * WL.dims.F * WL.dims.d * 2)) / r["gate_launches"]
        else:
            traffic = None
    ms_step = ms_max / args.steps
    a_cf = alpha_ref(args.mode, WL.n) if p is not None else None
    wgbs = r["wbytes"] / (r["ms"] / 1e3) / 1e9
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "committed tokens/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if WL.dims.dtype == "bf16" else "f32",
        "data": "synthetic (seeded random-init weights drawn on the GPU, uniform-random prompt ids)",
        "config": {"workload": f"{WL.name}: L{WL.dims.L} d{WL.dims.d} {WL.dims.Hq}q/{WL.dims.Hkv}kv x{WL.dims.hd} "
                               f"F{WL.dims.F} V{WL.dims.V}, n={WL.n}, Ls={WL.Ls}, "
                               f"anchors {','.join(str(a) for a in WL.anchors)}, prompt {WL.prompt_len}, {args.mode}"
                               + ("" if args.speculate == "input" else ", output-state schedule"),
                   "mode": args.mode, "n": WL.n, "prompt_len": WL.prompt_len, "max_new": r["max_new"],
                   "speculate": args.speculate,
                   "parallelism": f"replicas x{ws}", "l2": l2_note(r["wbytes"] / args.steps),
                   "alpha": round(r["alpha"], 4), "S0": round(r["alpha"] * WL.n, 3),
                   "tok_s_at_closed_form_alpha": None if a_cf is None else round(a_cf * 1e3 / ms_step, 2),
                   "closed_form_alpha": None if a_cf is None else round(a_cf, 4),
                   "prefill_ms": round(r["prefill_ms"], 3),
                   "weight_GBps": round(wgbs, 1),
                   "weight_frac_of_measured_hbm": round(wgbs / hbm, 4),
                   "weight_frac_of_nominal_hbm": round(wgbs / NOMINAL_HBM_GBS, 4),
                   "hbm_denominators_GBps": {"measured": hbm, "nominal": NOMINAL_HBM_GBS}},
        "roofline": {"kernel": "target gate/up GEMV (k_gemv EPI_GATEUP)", "bound": "hbm",
                     "timed": "CUDA events around each gate/up launch on its stream, in a second timed region of the "
                              "same workload",
                     "achieved": round(g_ach, 1), "peak": hbm, "unit": "GB/s", "frac": round(g_ach / hbm, 4),
                     "traffic": None if traffic is None else round(traffic), "peak_kind": f"hbm_gbs ({pk_kind})",
                     "launches": r["gate_launches"]},
        "clocks": r["clocks"],
        "e2e": None if args.skip_e2e else {
            "value": round(r["e2e_tokens"] / r["e2e_s"], 2), "unit": "generated tokens/s (prefill + decode, "
            "host buffers)", "h2d_bytes_per_step": round(4 * r["prompt_len"] / r["e2e_steps"], 3),
            "d2h_bytes_per_step": round((4 * WL.max_new + 32 * math.ceil(r["e2e_steps"] / 8)) / r["e2e_steps"], 3),
            "call": "spd_generate"},
        "gpu_launches": r["launches_per_step"] * args.steps,
    }
    if ws == 1 and not args.no_cpu_baseline:
        try:
            sps, commits, dt, _, cores = oracle_sample(12, args.mode)
            alpha = cpu_alpha(args.mode, WL.n, r["alpha"])
            line["cpu_baseline"] = {"value": round(sps * alpha, 4), "unit": "committed tokens/s", "cores": cores,
                                    "kind": "oracle",
                                    "sample": f"fp64 oracle, same shape and mode, n={WL.n}, 32-token prompt (prefill "
                                              f"untimed), 12 pipeline steps timed ({dt:.1f} s); tokens/s = steps/s x "
                                              f"alpha {alpha:.4f} ("
                                              + ("closed form" if alpha_ref(args.mode, WL.n) is not None
                                                 else "the GPU run's") + ")"}
        except MemoryError as ex:
            line["cpu_baseline"] = {"value": None, "unit": "committed tokens/s", "cores": os.cpu_count(),
                                    "kind": "oracle", "sample": f"not run: {ex}"}
    print(json.dumps(line), flush=True)


def _max_op():
    import torch.distributed as dist
    return dist.ReduceOp.MAX


def _sum_op():
    import torch.distributed as dist
    return dist.ReduceOp.SUM


def main_reference(args, ws, rank):
    """The oracle (plain fp64 CPU restatement of the method) on this arm's workload.  Each
    timed step is one pipeline step of the oracle; value = steps/s x the same alpha the
    GPU arm's cpu_baseline uses (closed form where one exists, else the oracle sample's
    own commit rate after the pipeline fill).  e2e: the workload's own prompt, prefill and steps timed together."""
    if rank != 0:
        return
    k = max(1, min(args.steps, 12))
    w = max(0, min(args.warmup, 2))
    if alpha_ref(args.mode, WL.n) is None:
        k = max(k, 2 * WL.n - w)   # no closed form: the sample must reach past the pipeline fill
    sps, commits, dt, _, cores = oracle_sample(k + w, args.mode)
    # commits per step after the first n - 1 steps (no token leaves before them)
    alpha = cpu_alpha(args.mode, WL.n, commits / max(1, k + w - (WL.n - 1)))
    value = sps * alpha
    e_sps, e_commits, e_dt, e_pf, _ = oracle_sample(4, args.mode, e2e=True)
    e2e_tokens = 1 + 4 * alpha
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "committed tokens/s", "n_gpus": 1,
        "steps": k, "warmup": w, "ms_per_step": round(1e3 / sps, 2), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{WL.name}: L{WL.dims.L} d{WL.dims.d} {WL.dims.Hq}q/{WL.dims.Hkv}kv x{WL.dims.hd} "
                               f"F{WL.dims.F} V{WL.dims.V}, n={WL.n}, Ls={WL.Ls}, "
                               f"anchors {','.join(str(a) for a in WL.anchors)}, prompt {WL.prompt_len}, {args.mode}",
                   "mode": args.mode, "n": WL.n},
        "cpu_baseline": {"value": round(value, 4), "unit": "committed tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"fp64 oracle, same shape and mode, n={WL.n}, 32-token prompt (prefill untimed), "
                                   f"{k + w} steps ({dt:.1f} s); tokens/s = steps/s x alpha {alpha:.4f}"},
        "e2e": {"value": round(e2e_tokens / (e_pf + e_dt), 4), "unit": "generated tokens/s (prefill + decode, host "
                "buffers)", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0,
                "sample": f"prompt {WL.prompt_len} prefilled ({e_pf:.1f} s) + 4 steps ({e_dt:.1f} s); tokens = 1 + "
                          f"4 x alpha"},
    }
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
