"""Benchmark of the lightning-indexer path: score -> top-512 -> sparse MQA.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

A step is one pass of the whole path over one 2048-token prefill chunk (default workload
prefill_8k: 2048 query tokens at positions 6144..8191, 2048 compressed rows, 64 indexer heads
x 128 dims, 64 attention heads x 512 dims, k_top = 512).  Inputs are synthetic (seeded), held
in HBM before the timed region; L2 is flushed (a 256 MiB write) before every timed step.

Printed (one JSON line, rank 0): the whole-job throughput in query tokens/s timed with CUDA
events on the launching stream, per-stage times, the dominant kernel against its roofline
(peaks from MEASURED_PEAKS.json), the same metric end to end through the C ABI with pinned
host buffers (copies inside the timed region), the oracle timed on the host cores as a
reported baseline, SM clocks sampled during the timed region, and the launch count.  A
"decode" object adds the 1M-context decode loop (256 single-token steps, 63 row appends) in
decode tokens/s, issued from the host and replayed as one CUDA graph.

With --impl reference the oracle (plain C, fp64) is timed instead, on a bounded sample of
the same workload per step.  Under torchrun (--gpus N), every rank runs its own chunk (the
path shards over query tokens with no exchange), the timed region is bracketed by barriers
and the slowest rank's time is used.
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
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "indexed query tokens/s (score+top-512+sparse attn) at 8k–64k ctx; % roofline"
UNIT = "query tokens/s"
DEFAULT_WORKLOAD = "prefill_8k"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(synth.WORKLOADS))
    ap.add_argument("--impl", default="ds4x", choices=["ds4x", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--host-chunks", type=int, default=0,
                    help="token sub-chunks of the host-buffer call in the e2e leg (0: the library's choice)")
    ap.add_argument("--no-decode", action="store_true", help="skip the 1M-context decode measurement")
    ap.add_argument("--no-compress", action="store_true", help="skip the compressor measurement")
    ap.add_argument("--decode-steps", type=int, default=256, help="decode steps per timed call (decode_1m)")
    ap.add_argument("--extra-workloads", default="prefill_32k,prefill_64k",
                    help="other prefill chunks measured into the line's 'workloads' object (comma list, '' = none)")
    ap.add_argument("--extra-steps", type=int, default=20, help="timed steps of each extra workload")
    ap.add_argument("--seed", type=int, default=0)
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(torch, dist, x: float, world: int, dev) -> float:
    """The largest of every rank's x (the slowest rank sets a step's time); x itself at N = 1."""
    if world <= 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world: int, units_per_rank: int, ms: float) -> float:
    """Whole-job units per second: every rank processes its own units in `ms` (max over ranks)."""
    return world * units_per_rank / (ms / 1e3)


L2_NOTE = "flushed before every timed step (256 MiB write)"


def parallelism(world: int) -> str:
    return f"dp{world} (independent chunks per GPU)" if world > 1 else "single GPU"


def workload_config(wl: synth.Workload, l2_note: str = L2_NOTE, world: int = 1) -> dict:
    return {
        "workload": f"{wl.name}: {wl.T} query tokens at positions {wl.pos0}..{wl.pos0 + wl.T - 1}, "
                    f"ratio {wl.ratio} -> {wl.S} compressed rows; indexer q[{wl.T},{wl.H},{wl.D}] fp16, "
                    f"k[{wl.S},{wl.D}] fp16, w[{wl.T},{wl.H}] fp16; top-{wl.k_top}; sparse MQA "
                    f"{wl.Hq} heads x {wl.Dkv} over kv[{wl.S},{wl.Dkv}] {wl.kv_dtype}",
        "T": wl.T, "S": wl.S, "H": wl.H, "D": wl.D, "ratio": wl.ratio, "k_top": wl.k_top,
        "Hq": wl.Hq, "Dkv": wl.Dkv, "kv_dtype": wl.kv_dtype, "seed": 0,
        "l2": l2_note, "parallelism": parallelism(world),
        **({"window": wl.window,
            "attention": f"local-plus-pooled: each token's top-{wl.k_top} pooled rows and the raw rows of its "
                         f"last {wl.window} positions in one softmax (kv_local[{wl.T + wl.window - 1},{wl.Dkv}])"}
           if wl.window > 0 else {}),
    }


def visible_rows(wl: synth.Workload) -> np.ndarray:
    p = wl.pos0 + np.arange(wl.T, dtype=np.int64)
    return np.minimum(wl.S, (p + 1) // wl.ratio)


def window_rows(wl: synth.Workload) -> np.ndarray:
    """Raw rows each token attends: its last `window` positions (none below 0)."""
    p = wl.pos0 + np.arange(wl.T, dtype=np.int64)
    return np.minimum(p + 1, wl.window) if wl.window > 0 else np.zeros(wl.T, dtype=np.int64)


def algorithmic(wl: synth.Workload) -> dict:
    nv = visible_rows(wl)
    scored = nv[nv > wl.k_top]
    sel = np.minimum(nv, wl.k_top) + window_rows(wl)
    return {
        # scoring: one multiply-add per (token, head, dim, visible row)
        "score_flops": float(2 * wl.H * wl.D * scored.sum()),
        # top-k: read every visible score once, write k_top indices per token
        "topk_bytes": float(4 * scored.sum() + 4 * wl.k_top * wl.T),
        # attention: two products of 2*Hq*Dkv flops per (token, attended row: pooled and window)
        "attn_flops": float(4 * wl.Hq * wl.Dkv * sel.sum()),
        "attn_gather_bytes": float(2 * wl.Dkv * sel.sum()),
    }


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def profiled_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on the current
    kernel source (a source hash is stored beside the counters)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    try:
        d = json.load(open(path))
        e = d[workload][kernel]
        src = os.path.join(ROOT, "deepseek_v4_sparse_gb300", "csrc", e["source"])
        h = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
        return float(e["dram_bytes_per_launch"]) if h == e["source_sha256_16"] else None
    except (KeyError, ValueError, OSError):
        return None


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        import tempfile
        fd, self.path = tempfile.mkstemp(prefix="ds4x_clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------- CPU oracle
def oracle_path(o, wl: synth.Workload, inp, sel):
    """The oracle's whole path on the tokens `sel` of the chunk."""
    if wl.window > 0:
        o.index_and_attend_local(inp.q[sel], inp.w[sel], inp.k, inp.positions[sel], inp.q_attn[sel], inp.kv,
                                 inp.kv_local, wl.kv_dtype, wl.S, wl.ratio, wl.k_top, inp.local_pos0, wl.window,
                                 wl.scale)
    else:
        o.index_and_attend(inp.q[sel], inp.w[sel], inp.k, inp.positions[sel], inp.q_attn[sel], inp.kv,
                           wl.kv_dtype, wl.S, wl.ratio, wl.k_top, wl.scale)


def cpu_baseline(wl: synth.Workload, inp, target_s: float = 12.0, first: int = 16):
    """The oracle as it stands (whole path, fp64, OpenMP over tokens) on a bounded sample of
    the workload's tokens; returns (tokens/s, threads, description)."""
    import oracle
    o = oracle.default()
    threads = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))

    def run(n):
        sel = np.linspace(0, wl.T - 1, n).astype(np.int64)
        t0 = time.perf_counter()
        oracle_path(o, wl, inp, sel)
        return time.perf_counter() - t0

    dt = run(first)
    n = int(min(wl.T, max(first, first * target_s / max(dt, 1e-3))))
    n = max(threads, (n // threads) * threads)
    n = min(n, wl.T)
    dt = run(n)
    return n / dt, threads, f"{n} of the {wl.T} tokens (evenly spaced), whole path, OpenMP {threads} threads"


def run_reference(args, wl):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    inp = synth.make_inputs(wl, seed=args.seed)
    import oracle
    o = oracle.default()
    threads = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
    per_step = max(threads, 16)
    rng = np.random.default_rng(0)

    def step():
        sel = np.sort(rng.choice(wl.T, per_step, replace=False))
        oracle_path(o, wl, inp, sel)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t0
    value = per_step * args.steps / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(wl, world=world),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": f"{per_step} random tokens of the {wl.T}-token chunk per step"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------------- stage rooflines
def stage_roofline(wl: synth.Workload, st_mean, peaks: dict):
    """Per-stage times, the dominant stage against its roofline, and every stage's rate."""
    alg = algorithmic(wl)
    stages = {"score_ms": float(st_mean[0]), "topk_ms": float(st_mean[1]), "attn_ms": float(st_mean[2])}
    dom = int(np.argmax(st_mean))
    if dom == 0:
        ach = alg["score_flops"] / (st_mean[0] / 1e3) / 1e12
        roof = {"kernel": "score_kernel (tcgen05)", "bound": "tensor", "achieved": ach, "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s", "algorithmic": alg["score_flops"], "traffic": profiled_traffic("score", wl.name)}
    elif dom == 1:
        ach = alg["topk_bytes"] / (st_mean[1] / 1e3) / 1e9
        roof = {"kernel": "top-k kernel", "bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "algorithmic": alg["topk_bytes"], "traffic": profiled_traffic("topk", wl.name)}
    else:
        ach = alg["attn_flops"] / (st_mean[2] / 1e3) / 1e12
        roof = {"kernel": "sparse_mqa_kernel (tcgen05)", "bound": "tensor", "achieved": ach,
                "peak": peaks["bf16_tflops"], "unit": "TFLOP/s", "algorithmic": alg["attn_flops"],
                "traffic": profiled_traffic("attn", wl.name)}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["peak_source"] = f"{peaks['source']} (burst)"
    others = {
        "score_tflops": alg["score_flops"] / (st_mean[0] / 1e3) / 1e12,
        "score_frac": alg["score_flops"] / (st_mean[0] / 1e3) / 1e12 / peaks["bf16_tflops"],
        "topk_gbs": alg["topk_bytes"] / (st_mean[1] / 1e3) / 1e9,
        "topk_frac": alg["topk_bytes"] / (st_mean[1] / 1e3) / 1e9 / peaks["hbm_gbs"],
        "attn_tflops": alg["attn_flops"] / (st_mean[2] / 1e3) / 1e12,
        "attn_frac": alg["attn_flops"] / (st_mean[2] / 1e3) / 1e12 / peaks["bf16_tflops"],
        "attn_gather_gbs": alg["attn_gather_bytes"] / (st_mean[2] / 1e3) / 1e9,
    }
    return stages, roof, others


def measure_prefill(ds4x, torch, dev, stream, wl: synth.Workload, seed: int, steps: int, peaks: dict, flush,
                    cpu: bool):
    """One more prefill chunk on this GPU, timed like the headline workload (inputs resident, L2
    flushed before every step, CUDA events on the launching stream): `steps` whole-path calls for
    the throughput, `steps` staged calls for the per-stage times, and the oracle on a bounded
    sample of the chunk's tokens on the host cores."""
    inp = synth.make_inputs(wl, seed=seed)
    kvt = torch.bfloat16 if wl.kv_dtype == "bf16" else torch.float16

    def d16(a, dt):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(dt)
    q, w, k = d16(inp.q, torch.float16), d16(inp.w, torch.float16), d16(inp.k, torch.float16)
    qa, kv = d16(inp.q_attn, kvt), d16(inp.kv, kvt)
    pos = torch.from_numpy(inp.positions.copy()).to(dev)
    T, S, k_top = wl.T, wl.S, wl.k_top
    scores = torch.empty((T, S), dtype=torch.float32, device=dev)
    idx = torch.empty((T, k_top), dtype=torch.int32, device=dev)
    out = torch.empty_like(qa)
    lse = torch.empty((T, wl.Hq), dtype=torch.float32, device=dev)
    ws = torch.empty((max(1, ds4x.workspace_bytes(T, S, k_top)),), dtype=torch.uint8, device=dev)
    tws_n = ds4x.topk_workspace_bytes(T, S, k_top)
    tws = torch.empty((tws_n,), dtype=torch.uint8, device=dev) if tws_n else None

    def fused():
        ds4x.index_and_attend(q, w, k, pos, qa, kv, wl.ratio, k_top, S=S, scale=wl.scale, indices=idx, out=out,
                              lse=lse, workspace=ws, stream=stream)

    def staged(ev):
        ev[0].record(stream)
        ds4x.indexer_score(q, w, k, pos, wl.ratio, scores=scores, S=S, stream=stream)
        ev[1].record(stream)
        ds4x.topk(scores, pos, S, wl.ratio, k_top, indices=idx, workspace=tws, stream=stream)
        ev[2].record(stream)
        ds4x.sparse_attn(qa, kv, idx, S=S, scale=wl.scale, out=out, lse=lse, stream=stream)
        ev[3].record(stream)

    for _ in range(3):
        fused()
        staged([torch.cuda.Event(enable_timing=True) for _ in range(4)])
    torch.cuda.synchronize()
    fev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    sev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
    for i in range(steps):
        flush.zero_()
        fev[i][0].record(stream)
        fused()
        fev[i][1].record(stream)
    for i in range(steps):
        flush.zero_()
        staged(sev[i])
    torch.cuda.synchronize()
    assert ds4x.device_status() == ds4x.OK, f"a bounded device wait timed out ({wl.name})"
    ms = float(np.mean([a.elapsed_time(b) for a, b in fev]))
    st = np.array([[e[j].elapsed_time(e[j + 1]) for j in range(3)] for e in sev]).mean(axis=0)
    stages, roof, rates = stage_roofline(wl, st, peaks)
    res = {"config": workload_config(wl), "value": T / (ms / 1e3), "unit": UNIT, "ms_per_step": ms,
           "steps": steps, "warmup": 3, "roofline": roof, "stage_ms": stages, "stage_rates": rates,
           "staged_ms_per_step": float(st.sum())}
    if cpu:
        v, cores, desc = cpu_baseline(wl, inp, target_s=5.0, first=16)
        res["cpu_baseline"] = {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc}
    return res


# ---------------------------------------------------------------------------- decode loop
def measure_decode(ds4x, torch, dev, stream, seed: int, reps: int = 3, n_steps: int = 256, warm: int = 1,
                   window: int = 0):
    """The 1M-context decode: n_steps single-token steps from position 1048575 over 262144
    resident rows, a row appended every 4 positions (63 over 256 steps), each step
    score -> top-512 -> sparse MQA.  One timed unit is a whole ds4x_decode call (appends
    included), L2 flushed before it; reported as issued from the host and as one CUDA-graph
    replay of the same call, plus a per-kernel split of one step."""
    wl = synth.WORKLOADS["decode_1m"]
    S0 = wl.S
    inp = synth.make_inputs(wl, seed=seed, T=n_steps, S=S0)
    kvt = torch.bfloat16 if wl.kv_dtype == "bf16" else torch.float16

    def dev16(a, dt):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(dt)

    q, w, qa = dev16(inp.q, torch.float16), dev16(inp.w, torch.float16), dev16(inp.q_attn, kvt)
    k, kv = dev16(inp.k, torch.float16), dev16(inp.kv, kvt)          # capacity rows
    k_new, kv_new = k[S0:].clone(), kv[S0:].clone()                   # the rows the loop appends
    cap = k.shape[0]
    pos = torch.empty((n_steps,), dtype=torch.int32, device=dev)
    idx = torch.empty((n_steps, wl.k_top), dtype=torch.int32, device=dev)
    out = torch.empty_like(qa)
    lse = torch.empty((n_steps, wl.Hq), dtype=torch.float32, device=dev)
    ws = torch.empty((ds4x.decode_local_workspace_bytes(cap, wl.k_top, window),), dtype=torch.uint8, device=dev)
    flush = torch.empty((256 << 20,), dtype=torch.uint8, device=dev)
    if window > 0:
        # raw rows of every position up to the last step: the window's history and the steps' own
        raw_cap = wl.pos0 + n_steps
        kv_raw = torch.zeros((raw_cap, wl.Dkv), dtype=kvt, device=dev)
        kv_raw[wl.pos0 - window:wl.pos0] = dev16(synth.local_rows(seed, "bench_decode_raw", window, wl.Dkv, "normal",
                                                                  wl.kv_dtype), kvt)
        kv_raw_new = dev16(synth.local_rows(seed, "bench_decode_raw_new", n_steps, wl.Dkv, "normal", wl.kv_dtype), kvt)

    def launch(st):
        if window > 0:
            return ds4x.decode_local(q, w, qa, k, kv, S0, wl.pos0, wl.ratio, kv_raw, kv_raw_new, window, k_new=k_new,
                                     kv_new=kv_new, k_top=wl.k_top, scale=wl.scale, positions=pos, indices=idx,
                                     out=out, lse=lse, workspace=ws, stream=st)
        return ds4x.decode(q, w, qa, k, kv, S0, wl.pos0, wl.ratio, k_new=k_new, kv_new=kv_new, k_top=wl.k_top,
                           scale=wl.scale, positions=pos, indices=idx, out=out, lse=lse, workspace=ws, stream=st)

    def call():
        r = launch(stream)
        return r[4], ds4x.last_launch_count()

    for _ in range(max(1, warm)):
        s_final, launches = call()
    torch.cuda.synchronize()
    assert ds4x.device_status() == ds4x.OK
    times = []
    for _ in range(reps):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        call()
        e1.record(stream)
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
    ms = float(np.median(times))
    # the same call captured once into a CUDA graph and replayed
    graph_ms = None
    try:
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            with torch.cuda.graph(g, stream=side):
                launch(side)
        stream.wait_stream(side)
        gt = []
        for _ in range(reps):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            g.replay()
            e1.record(stream)
            torch.cuda.synchronize()
            gt.append(e0.elapsed_time(e1))
        graph_ms = float(np.median(gt))
        assert ds4x.device_status() == ds4x.OK
    except RuntimeError as e:  # capture refused: report the host-issued number only
        graph_ms = None
        print(f"decode graph capture unavailable: {e}", file=sys.stderr)
    if window > 0:
        return {
            "workload": f"decode_1m with a {window}-position raw window: {n_steps} steps of 1 query token at positions "
                        f"{wl.pos0}..{wl.pos0 + n_steps - 1}, each attending to its top-{wl.k_top} pooled rows and "
                        f"the raw rows of its last {window} positions (ds4x_decode_local)",
            "value": n_steps / (ms / 1e3), "unit": "decode tokens/s", "us_per_step": 1e3 * ms / n_steps,
            "graph_value": None if graph_ms is None else n_steps / (graph_ms / 1e3),
            "graph_us_per_step": None if graph_ms is None else 1e3 * graph_ms / n_steps,
            "steps": n_steps, "gpu_launches_per_call": int(launches),
        }
    # per-kernel split of the last step (T = 1 over S_final rows), each stage timed alone
    S = s_final
    sc = torch.empty((1, S), dtype=torch.float32, device=dev)
    tws = torch.empty((max(16, ds4x.topk_workspace_bytes(1, S, wl.k_top)),), dtype=torch.uint8, device=dev)
    i = n_steps - 1
    p_last = pos[i:i + 1].clone()          # a 16-byte aligned copy of the step's position
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    split = []
    for _ in range(reps):
        flush.zero_()
        ev[0].record(stream)
        ds4x.indexer_score(q[i:i + 1], w[i:i + 1], k, p_last, wl.ratio, scores=sc, S=S, stream=stream)
        ev[1].record(stream)
        ds4x.topk(sc, p_last, S, wl.ratio, wl.k_top, indices=idx[i:i + 1], workspace=tws, stream=stream)
        ev[2].record(stream)
        ds4x.index_and_attend(q[i:i + 1], w[i:i + 1], k, p_last, qa[i:i + 1], kv, wl.ratio, wl.k_top, S=S,
                              scale=wl.scale, indices=idx[i:i + 1], out=out[i:i + 1], lse=lse[i:i + 1],
                              workspace=ws, stream=stream)
        ev[3].record(stream)
        torch.cuda.synchronize()
        split.append([ev[j].elapsed_time(ev[j + 1]) * 1e3 for j in range(3)])
    sp = np.median(np.array(split), axis=0)
    return {
        "workload": f"decode_1m: {n_steps} steps of 1 query token at positions {wl.pos0}..{wl.pos0 + n_steps - 1}, "
                    f"ratio {wl.ratio}, {S0} resident rows + {s_final - S0} appended (capacity {cap}); "
                    f"k[{cap},{wl.D}] fp16, kv[{cap},{wl.Dkv}] {wl.kv_dtype}; top-{wl.k_top}",
        "value": n_steps / (ms / 1e3), "unit": "decode tokens/s", "us_per_step": 1e3 * ms / n_steps,
        "graph_value": None if graph_ms is None else n_steps / (graph_ms / 1e3),
        "graph_us_per_step": None if graph_ms is None else 1e3 * graph_ms / n_steps,
        "steps": n_steps, "appended_rows": int(s_final - S0), "gpu_launches_per_call": int(launches),
        "l2": "flushed before every timed call; within a call the steps re-read k from L2 as a decode does",
        "one_step_us": {"score": float(sp[0]), "topk": float(sp[1]), "fused_step": float(sp[2])},
    }


def measure_compress(ds4x, torch, dev, stream, seed: int, reps: int = 20):
    """The compressor on a 2048-token prefill chunk (k rows: fp16 D=128; kv rows: bf16 D=512; ratio 4
    and 128, a 3-position frontier held over) and on a 64k-token batch of kv rows (HBM bandwidth).
    Device time per call, L2 flushed before each; bytes = every input byte once + the outputs."""
    flush = torch.empty((256 << 20,), dtype=torch.uint8, device=dev)
    cases = [("k_8k_r4", "f16", 128, 4, 2048, 3), ("kv_8k_r4", "bf16", 512, 4, 2048, 3),
             ("kv_8k_r128", "bf16", 512, 128, 2048, 3), ("kv_64k_r4", "bf16", 512, 4, 65536, 3)]
    out = {}
    for name, dt, D, ratio, T, f in cases:
        x, g, fx, fg, bias = synth.compress_inputs(seed, f"bench_{name}", T, D, ratio, dt, f)
        tdt = torch.bfloat16 if dt == "bf16" else torch.float16

        def d16(a):
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(tdt)
        dx, dg, dfx, dfg = d16(x), d16(g), d16(fx), d16(fg)
        db = torch.from_numpy(bias).to(dev)
        n_out, rem = (f + T) // ratio, (f + T) % ratio
        rows = torch.empty((n_out, D), dtype=tdt, device=dev)
        fxo = torch.empty((max(rem, 1), D), dtype=tdt, device=dev)
        fgo = torch.empty((max(rem, 1), D), dtype=tdt, device=dev)
        ts = []
        for i in range(reps + 3):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            ds4x.compress(dx, dg, db, ratio, dfx, dfg, rows=rows, frontier_x_out=fxo, frontier_g_out=fgo,
                          stream=stream)
            e1.record(stream)
            if i >= 3:
                ts.append((e0, e1))
        torch.cuda.synchronize()
        us = float(np.median([a.elapsed_time(b) for a, b in ts])) * 1e3
        nbytes = 2 * (f + T) * D * 2 + ratio * D * 4 + n_out * D * 2 + 2 * rem * D * 2
        out[name] = {"T": T, "D": D, "ratio": ratio, "dtype": dt, "us": us, "bytes": nbytes,
                     "gbs": nbytes / (us * 1e-6) / 1e9}
    return out


def decode_roofline(dec: dict, peaks: dict) -> dict:
    """A decode step is bound by memory: every step reads all of k ([rows, 128] fp16) for the scores,
    writes and reads one fp32 score per row, and gathers 512 kv rows; rows = the call's average S."""
    wl = synth.WORKLOADS["decode_1m"]
    rows = wl.S + dec["appended_rows"] / 2.0
    step_bytes = 2.0 * wl.D * rows + 2 * 4.0 * rows + 2.0 * wl.Dkv * wl.k_top
    roof = {"kernel": "decode step (score, top-k, attention launches)", "bound": "hbm",
            "achieved": step_bytes / (dec["us_per_step"] * 1e-6) / 1e9, "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "algorithmic": step_bytes, "traffic": None}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["peak_source"] = f"{peaks['source']} (burst)"
    if dec.get("graph_us_per_step"):
        roof["graph_frac"] = step_bytes / (dec["graph_us_per_step"] * 1e-6) / 1e9 / peaks["hbm_gbs"]
    return roof


def decode_main(args, ds4x, torch, dev, rank, world):
    """--workload decode_1m: the decode loop is the step (one call = decode_steps tokens)."""
    import torch.distributed as dist
    stream = torch.cuda.current_stream()
    sampler = ClockSampler(dev.index or 0)
    with sampler:
        dec = measure_decode(ds4x, torch, dev, stream, args.seed + rank, reps=max(1, args.steps),
                             n_steps=args.decode_steps, warm=max(3, args.warmup))
    peaks = load_peaks()
    roof = decode_roofline(dec, peaks)
    # the slowest rank's time per decode step; each rank decodes its own token stream
    us_step = max_over_ranks(torch, dist, dec["us_per_step"], world, dev)
    if rank == 0:
        step_ms = 1e3 * dec["steps"] / dec["value"]
        line = {
            "metric": METRIC, "value": job_throughput(world, 1, us_step / 1e3), "unit": "decode tokens/s",
            "n_gpus": world,
            "steps": max(1, args.steps), "warmup": max(3, args.warmup), "ms_per_step": step_ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16+bf16 (fp32 accumulate)",
            "data": "synthetic", "config": {"workload": dec["workload"], "l2": dec["l2"]},
            "roofline": roof, "decode": dec, "cpu_baseline": None, "e2e": None,
            "gpu_launches": dec["gpu_launches_per_call"] * max(1, args.steps), "clocks": sampler.summary(),
        }
        print(json.dumps(line), flush=True)


# ------------------------------------------------------------------------------- GPU arm
def main():
    args = parse()
    wl = synth.WORKLOADS[args.workload]
    if args.impl == "reference":
        return run_reference(args, wl)

    import torch
    import torch.distributed as dist

    import deepseek_v4_sparse_gb300 as ds4x
    from deepseek_v4_sparse_gb300 import build as ds4x_build

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0 or not os.path.exists(ds4x.LIB_PATH):
        ds4x_build.build()
    if world > 1:
        dist.barrier()
    ds4x.load()

    if wl.name == "decode_1m":
        return decode_main(args, ds4x, torch, dev, rank, world)

    # every rank processes its own chunk: same shapes, its own seed
    inp = synth.make_inputs(wl, seed=args.seed + rank)
    # inputs on the host (pinned, for the end-to-end leg) and on the device
    def pinned16(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).pin_memory()
    h = {"q": pinned16(inp.q), "w": pinned16(inp.w), "k": pinned16(inp.k), "q_attn": pinned16(inp.q_attn),
         "kv": pinned16(inp.kv), "positions": torch.from_numpy(inp.positions.copy()).pin_memory()}
    win = wl.window > 0
    if win:
        h["kv_local"] = pinned16(inp.kv_local)
    kvt = torch.bfloat16 if wl.kv_dtype == "bf16" else torch.float16
    dt_of = {"q": torch.float16, "w": torch.float16, "k": torch.float16, "q_attn": kvt, "kv": kvt,
             "positions": torch.int32, "kv_local": kvt}
    d = {n: h[n].to(dev).view(dt_of[n]) for n in h}
    T, S, k_top = wl.T, wl.S, wl.k_top
    scores = torch.empty((T, S), dtype=torch.float32, device=dev)
    idx = torch.empty((T, k_top), dtype=torch.int32, device=dev)
    cnt = torch.empty((T,), dtype=torch.int32, device=dev)
    out = torch.empty_like(d["q_attn"])
    lse = torch.empty((T, wl.Hq), dtype=torch.float32, device=dev)
    ws = torch.empty((max(1, ds4x.workspace_bytes_local(T, S, k_top, wl.window)),), dtype=torch.uint8, device=dev)
    tws_n = ds4x.topk_workspace_bytes(T, S, k_top)
    tws = torch.empty((max(1, tws_n),), dtype=torch.uint8, device=dev) if tws_n else None
    flush = torch.empty((256 << 20,), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def fused():
        if win:
            ds4x.index_and_attend_local(d["q"], d["w"], d["k"], d["positions"], d["q_attn"], d["kv"], d["kv_local"],
                                        wl.ratio, inp.local_pos0, wl.window, k_top, S=S, scale=wl.scale,
                                        indices=idx, out=out, lse=lse, workspace=ws, stream=stream)
        else:
            ds4x.index_and_attend(d["q"], d["w"], d["k"], d["positions"], d["q_attn"], d["kv"], wl.ratio, k_top,
                                  S=S, scale=wl.scale, indices=idx, out=out, lse=lse, workspace=ws, stream=stream)
        return ds4x.last_launch_count()

    def staged(ev):
        ev[0].record(stream)
        ds4x.indexer_score(d["q"], d["w"], d["k"], d["positions"], wl.ratio, scores=scores, S=S, stream=stream)
        n = ds4x.last_launch_count()
        ev[1].record(stream)
        ds4x.topk(scores, d["positions"], S, wl.ratio, k_top, indices=idx, counts=cnt, workspace=tws,
                  stream=stream)
        n += ds4x.last_launch_count()
        ev[2].record(stream)
        if win:
            ds4x.local_pooled_attn(d["q_attn"], d["kv"], d["kv_local"], idx, d["positions"], inp.local_pos0,
                                   wl.window, S=S, scale=wl.scale, out=out, lse=lse, stream=stream)
        else:
            ds4x.sparse_attn(d["q_attn"], d["kv"], idx, S=S, scale=wl.scale, out=out, lse=lse, stream=stream)
        n += ds4x.last_launch_count()
        ev[3].record(stream)
        return n

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    # ---------------------------------------------------------------- warm-up
    for _ in range(max(3, args.warmup)):
        fused()
        staged([torch.cuda.Event(enable_timing=True) for _ in range(4)])
    torch.cuda.synchronize()
    assert ds4x.device_status() == ds4x.OK, "a bounded device wait timed out during warm-up"

    # ------------------------------------------------- timed region (device-resident)
    launches = 0
    sampler = ClockSampler(local)
    with sampler:
        barrier()
        fused_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                    for _ in range(args.steps)]
        stage_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
        for i in range(args.steps):
            flush.zero_()
            fused_ev[i][0].record(stream)
            launches += fused()
            fused_ev[i][1].record(stream)
        for i in range(args.steps):
            flush.zero_()
            launches += staged(stage_ev[i])
        barrier()
    fused_ms = [a.elapsed_time(b) for a, b in fused_ev]
    stage_ms = np.array([[e[j].elapsed_time(e[j + 1]) for j in range(3)] for e in stage_ev])
    step_ms = max_over_ranks(torch, dist, float(np.mean(fused_ms)), world, dev)
    assert ds4x.device_status() == ds4x.OK, "a bounded device wait timed out during the timed region"

    # ------------------------------------------- end to end through the C ABI (host buffers)
    e2e = None
    if not args.no_e2e:
        h_out = torch.empty(out.shape, dtype=torch.int16).pin_memory()
        h_idx = torch.empty(idx.shape, dtype=torch.int32).pin_memory()
        h_lse = torch.empty(lse.shape, dtype=torch.float32).pin_memory()
        h2d = sum(h[n].numel() * h[n].element_size() for n in h)
        d2h = h_out.numel() * 2 + h_idx.numel() * 4 + h_lse.numel() * 4
        e_steps = max(5, min(args.steps, 11))
        # the public host-buffer call: it copies the inputs in, runs the path and copies the
        # outputs back, overlapping the copies with the work by sub-chunks of tokens
        hv = {n: h[n].view(dt_of[n]) for n in h}
        L = inp.kv_local.shape[0] if win else 0
        hbuf = torch.empty((ds4x.index_and_attend_local_host_bytes(T, wl.H, wl.D, S, k_top, wl.Hq, wl.Dkv, L,
                                                                   wl.window, args.host_chunks),),
                           dtype=torch.uint8, device=dev)

        def e2e_step():
            if win:
                ds4x.index_and_attend_local_host(hv["q"], hv["w"], hv["k"], hv["positions"], hv["q_attn"], hv["kv"],
                                                 hv["kv_local"], wl.ratio, inp.local_pos0, wl.window, k_top, S=S,
                                                 scale=wl.scale, n_chunks=args.host_chunks, indices=h_idx, out=h_out,
                                                 lse=h_lse, device_buffer=hbuf, stream=stream)
            else:
                ds4x.index_and_attend_host(hv["q"], hv["w"], hv["k"], hv["positions"], hv["q_attn"], hv["kv"],
                                           wl.ratio, k_top, S=S, scale=wl.scale, n_chunks=args.host_chunks,
                                           indices=h_idx, out=h_out, lse=h_lse, device_buffer=hbuf, stream=stream)

        e2e_step()
        barrier()
        # a step is the interval between marks recorded on the stream before and after each call
        # (the call's copies start after the first and the stream waits for its last copy out);
        # the median step is reported: the host link is shared with the machine's other GPUs
        marks = [torch.cuda.Event(enable_timing=True) for _ in range(e_steps + 1)]
        marks[0].record(stream)
        for i in range(e_steps):
            e2e_step()
            marks[i + 1].record(stream)
        barrier()
        per_step = [marks[i].elapsed_time(marks[i + 1]) for i in range(e_steps)]
        e_ms = max_over_ranks(torch, dist, float(np.median(per_step)), world, dev)
        e2e = {"value": job_throughput(world, T, e_ms), "unit": UNIT, "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(d2h), "ms_per_step": e_ms, "steps": e_steps,
               "ms_per_step_min_max": [float(min(per_step)), float(max(per_step))],
               "call": ("ds4x_index_and_attend_local_host" if win else "ds4x_index_and_attend_host") +
                       " (page-locked host buffers; copies in, work and copies out "
                       "overlapped by sub-chunks of tokens)", "host_chunks": args.host_chunks}

    # ------------------------------------------------------------------ roofline
    peaks = load_peaks()
    st_mean = stage_ms.mean(axis=0)
    stages, roof, others = stage_roofline(wl, st_mean, peaks)

    dec = dec_local = None
    if rank == 0 and not args.no_decode and wl.name != "decode_1m":
        dec = measure_decode(ds4x, torch, dev, stream, args.seed)
        dec["roofline"] = decode_roofline(dec, peaks)
        dec_local = measure_decode(ds4x, torch, dev, stream, args.seed, window=128)

    extra = None
    names = [n for n in args.extra_workloads.split(",") if n and n != wl.name]
    if rank == 0 and names:
        extra = {n: measure_prefill(ds4x, torch, dev, stream, synth.WORKLOADS[n], args.seed, args.extra_steps,
                                    peaks, flush, cpu=not args.no_cpu_baseline and world == 1)
                 for n in names}

    comp = None
    if rank == 0 and not args.no_compress:
        comp = measure_compress(ds4x, torch, dev, stream, args.seed)
        for v in comp.values():
            v["hbm_frac"] = v["gbs"] / peaks["hbm_gbs"]

    cpu = None
    if rank == 0 and not args.no_cpu_baseline and world == 1:
        v, cores, desc = cpu_baseline(wl, inp)
        cpu = {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc}

    if rank == 0:
        line = {
            "metric": METRIC, "value": job_throughput(world, T, step_ms), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f16+bf16 (fp32 accumulate)",
            "data": "synthetic",
            "config": workload_config(wl, world=world),
            "roofline": roof, "stage_ms": stages, "stage_rates": others,
            "staged_ms_per_step": float(stage_ms.sum(axis=1).mean()),
            "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": int(launches),
            "clocks": sampler.summary(), "workloads": extra, "decode": dec, "decode_local": dec_local,
            "compress": comp,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
