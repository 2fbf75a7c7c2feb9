"""Throughput of the DeepSeekMoE layer forward on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--preset NAME] [--tokens T] [--experts E]

A step is one moe_layer_forward over one batch of T tokens: router GEMM,
sigmoid, group-limited top-K, load count, scan, permutation, grouped SwiGLU
expert GEMMs, shared expert with the fused gate-weighted combine, and the
+/- gamma bias update. Inputs are seeded synthetic tensors already resident
in HBM (x 235 MB and 22.5 GB of weights at the default V3 shape, both larger
than L2, so no flush is needed between steps). Rank 0 prints one JSON line.

--impl reference times the CPU oracle (the plain float64 restatement of the
layer under oracle/) on the host cores on a bounded sample of the same
workload and prints the same kind of line with "impl": "reference".
"""
from __future__ import annotations

import argparse
import datetime
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from mixture_experts_layer_100_b300 import synth  # noqa: E402

METRIC = "MoE-layer tokens/sec (1×B300, V3 shape T=16K bf16); % tensor/HBM roofline"
DEFAULT_PRESET = "v3_t16384_d7168_e256_bf16"
L2_BYTES = 126 * 2 ** 20
STAGES = ["router_gemm", "route_select", "permute", "gemm1_swiglu", "gemm2_routed", "gemm2_shared_combine",
          "bias_update"]


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--preset", default=DEFAULT_PRESET)
    ap.add_argument("--tokens", type=int, default=None)
    ap.add_argument("--experts", type=int, default=None)
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="skip the CUDA-graph replay timing")
    ap.add_argument("--no-standalone", action="store_true",
                    help="skip the standalone timing of moe_route / moe_permute")
    ap.add_argument("--combine", choices=["gather", "scatter_add"], default=None,
                    help="moe_layer_forward's combine mode (default: the workload's)")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the decode-shape and FP8 workloads timed after the V3 bf16 headline")
    return ap.parse_args()


def preset_from_args(a):
    p = synth.PRESETS[a.preset]
    if a.combine is not None:
        p = p.replace(combine=a.combine)
    if a.tokens is not None:
        p = p.replace(T=a.tokens)
    if a.experts is not None:
        p = p.replace(E=a.experts)
    return p


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            m = json.load(f)
        return m["hbm_gbs"], m["bf16_tflops"], m["bf16_tflops_sustained"], "measured"
    except Exception:
        return 6400.0, 1800.0, 1400.0, "fallback"


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clocks, power and throttle reasons every 50 ms. The sampler
    is started before the timed region and waits (up to 3 s) for its first
    sample; mark(start/end) bracket the timed region on the host clock, and
    summary() keeps the samples taken inside it (all samples if none)."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int, enabled: bool = True):
        self.enabled = enabled
        self.idx = device_index
        self.proc = None
        self.t0 = self.t1 = None

    def __enter__(self):
        if not self.enabled:
            return self
        self.tmp = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=self.tmp, stderr=subprocess.DEVNULL)
        except FileNotFoundError:
            self.proc = None
            return self
        deadline = time.time() + 3.0
        while time.time() < deadline and os.path.getsize(self.tmp.name) == 0:
            time.sleep(0.02)
        return self

    def mark_start(self):
        self.t0 = datetime.datetime.now()

    def mark_end(self):
        self.t1 = datetime.datetime.now()

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    @staticmethod
    def parse(lines, t0=None, t1=None):
        """Samples of nvidia-smi csv lines (FIELDS order) -> summary dict;
        only those stamped within [t0, t1] when any are."""
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        rows = []
        for line in lines:
            f = [v.strip() for v in line.split(",")]
            if len(f) < 10:
                continue
            try:
                sm, mx = float(f[2]), float(f[3])
            except ValueError:
                continue
            try:
                ts = datetime.datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f")
            except ValueError:
                ts = None  # unknown stamp format: the sample counts only among all samples
            try:
                pw = float(f[4])
            except ValueError:
                pw = None
            rows.append((ts, sm, mx, pw, [n for n, v in zip(names, f[6:10]) if v.lower().startswith("active")]))
        if not rows:
            return None
        inside = [r for r in rows if None not in (t0, t1, r[0]) and t0 <= r[0] <= t1]
        use = inside or rows
        pws = [r[3] for r in use if r[3] is not None]
        return {"sm_mhz": statistics.median(r[1] for r in use), "sm_max_mhz": max(r[2] for r in use),
                "reasons": sorted({n for r in use for n in r[4]}), "samples": len(use),
                "samples_in_timed_region": len(inside),
                "power_w_median": statistics.median(pws) if pws else None}

    def summary(self):
        if self.proc is None:
            return None
        self.tmp.flush()
        self.tmp.seek(0)
        lines = self.tmp.read().strip().splitlines()
        os.unlink(self.tmp.name)
        return self.parse(lines, self.t0, self.t1)


# ---------------------------------------------------------------- helpers
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


# kernel and launch sources that the roofline kernel's recorded DRAM traffic
# depends on, per expert-GEMM dtype (profiles/traffic.json, key
# "gemm1_swiglu:<dtype>")
TRAFFIC_SOURCES = {
    "bf16": ("gemm_tc.cu", "gemm_epi.cuh", "gemm_sched.cuh", "stages.cu"),
    "e4m3": ("gemm_fp8.cu", "gemm_fp8.cuh", "gemm_sched.cuh", "stages.cu"),
    "e4m3_ue8m0": ("gemm_mx.cu", "gemm_fp8.cuh", "gemm_sched.cuh", "stages.cu"),
}


def source_sha(files) -> str:
    """Hash of the kernel and launch sources a traffic measurement depends on."""
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "mixture_experts_layer_100_b300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def traffic_from_profiles(stage: str, dtype: str):
    """DRAM bytes per launch recorded in profiles/ for this stage's kernel at
    the given expert dtype, if its kernel and launch sources are unchanged
    since the capture (else None)."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            rec = json.load(f)[f"{stage}:{dtype}"]
        ok = rec.get("source_sha") == source_sha(TRAFFIC_SOURCES[dtype])
        return rec["bytes_per_launch"] if ok else None
    except Exception:
        return None


def flops_gemm1(p):
    """Routed experts' GEMM1 (the shared experts' GEMM1 runs on a side stream,
    overlapped with routing and permutation, and is not in this stage)."""
    return 2.0 * p.T * p.K * p.d * 2 * p.I


def flops_gemm2_routed(p):
    return 2.0 * p.T * p.K * p.I * p.d


def flops_gemm2_shared(p):
    return 2.0 * p.T * p.S * p.I * p.d


def hbm_bytes(p):
    """Algorithmic DRAM bytes per step of the memory-bound stages."""
    a = 2 if p.dtype == "bf16" else 4
    return {
        "router_gemm": p.T * p.d * a + p.E * p.d * a + p.T * p.E * 4,
        "route_select": p.T * p.E * 4 + p.T * p.K * 8,
        "permute": p.T * p.d * a + p.T * p.K * p.d * a + p.T * p.K * 16,
        # routed sum: K gathered rows in, r out; epilogue: r in, out written
        "gemm2_shared_combine": p.T * p.K * p.d * a + 3 * p.T * p.d * a + p.T * p.K * 8,
    }


# ---------------------------------------------------------------- CPU oracle leg
class CpuOracleUnit:
    """One bounded unit of the workload run by the C++ CPU oracle
    (oracle/moe_oracle.cpp, plain loops in double, g++ -O2) on the host cores:
    the routing of a block of `nt` tokens (router GEMM and sigmoid,
    group-limited top-K, load count, bias update) and the SwiGLU FFN of the
    block's first `rows` tokens on two experts (the first shared expert, or
    routed expert 0 when S = 0, and the routed expert E/2), in the workload's
    expert precision. Tokens/s is extrapolated as
    1 / (t_route / nt + (K + S) * t_ffn / (2 * rows)): every token runs K
    routed and S shared expert FFNs of the same cost. Both the bench line's
    cpu_baseline and the reference arm time this unit. Host copies of the
    inputs are made once, untimed."""

    def __init__(self, p, w, x_host, nt=4096, rows=128):
        import numpy as np
        self.p = p
        self.nt = min(nt, p.T)
        self.rows = min(rows, self.nt)
        self.xb = np.ascontiguousarray(x_host[:self.nt].float().numpy())
        self.wr = w.w_router.float().cpu().numpy()
        self.b = synth.make_bias(p).numpy()
        first = (w.ws13[0], w.ws2[0]) if p.S > 0 else (w.w13[0], w.w2[0])
        self.ew = [(first[0].float().cpu().numpy(), first[1].float().cpu().numpy()),
                   (w.w13[p.E // 2].float().cpu().numpy(), w.w2[p.E // 2].float().cpu().numpy())]
        self.f8 = p.expert_dtype in ("e4m3", "e4m3_ue8m0")
        self.desc = (f"C++ oracle: routing + load count + bias update of {self.nt} tokens, and the "
                     f"{p.expert_dtype} SwiGLU FFN of {self.rows} tokens on 2 experts, extrapolated to "
                     f"K+S={p.K + p.S} expert FFNs per token")

    def run(self):
        """Returns (tokens/s extrapolated to the whole layer, seconds)."""
        import numpy as np
        from oracle import cpp
        p = self.p
        t0 = time.perf_counter()
        s = cpp.router_scores(self.xb, self.wr)
        idx, _ = cpp.select_experts(s, self.b, p.G, p.K, p.M, p.group_topk)
        cpp.bias_update(cpp.expert_counts(idx, p.E), self.b, p.gamma, self.nt, p.K)
        t1 = time.perf_counter()
        acc = np.zeros((self.rows, p.d))
        for w13, w2 in self.ew:
            cpp.expert_accumulate(self.xb[:self.rows], np.arange(self.rows), w13, w2, None, acc, fp8=self.f8,
                                  ue8m0=p.expert_dtype == "e4m3_ue8m0")
        t2 = time.perf_counter()
        per_tok = (t1 - t0) / self.nt + (p.K + p.S) * (t2 - t1) / (len(self.ew) * self.rows)
        return 1.0 / per_tok, t2 - t0

    @staticmethod
    def cores():
        """Threads the C++ oracle runs on: std::thread::hardware_concurrency()."""
        from oracle import cpp
        return cpp.hardware_threads()


def bench_config(p, world):
    """The `config` object of both arms' JSON lines."""
    return {"workload": p.name, "T": p.T, "d": p.d, "E": p.E, "G": p.G, "K": p.K, "M": p.M, "I": p.I, "S": p.S,
            "gamma": p.gamma, "global_tokens_per_step": p.T * world,
            "parallelism": f"dp{world} replicas" if world > 1 else "single GPU",
            "l2": l2_note(p), "combine": p.combine,
            "zipf_alpha": synth.ZIPF_ALPHA if p.zipf else None}


def l2_note(p):
    a = 2 if p.dtype == "bf16" else 4
    xb, wb = p.T * p.d * a, (p.E + p.S) * 3 * p.d * p.I * a
    big = xb > L2_BYTES and wb > L2_BYTES
    return (f"x {xb / 1e6:.0f} MB, weights {wb / 1e9:.2f} GB: " +
            ("inputs larger than L2, no flush" if big else "weights larger than L2, no flush"
             if wb > L2_BYTES else "smaller than L2 (parity-size workload)"))


def run_reference(a, p):
    world, rank, local = dist_env()
    if rank != 0:
        return
    dev = f"cuda:{local}" if torch.cuda.is_available() else "cpu"
    w = synth.make_weights(p, device=dev)
    x = synth.make_x(p, w.w_router, device=dev).cpu()
    unit = CpuOracleUnit(p, w, x)
    del w
    for _ in range(a.warmup):
        unit.run()
    vals, secs = [], 0.0
    for _ in range(a.steps):
        v, s = unit.run()
        vals.append(v)
        secs += s
    value = a.steps / sum(1.0 / v for v in vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": a.gpus,
        "steps": a.steps, "warmup": a.warmup, "ms_per_step": 1000.0 * secs / a.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": bench_config(p, a.gpus),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": CpuOracleUnit.cores(), "kind": "oracle",
                         "sample": unit.desc + " (one unit per step)"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- end to end
def run_e2e(a, p, x, out, step, dev, pg):
    """The same step fed from pinned host memory: every step copies its batch
    host -> device and its output device -> host. Batches are double-buffered
    over three streams (input copies, compute, output copies), so the copies of
    batch i+1 and i-1 overlap the layer on batch i, as in a serving loop."""
    n = min(a.e2e_steps, a.steps)
    xh = x.cpu().pin_memory()
    oh = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
    xd = [torch.empty_like(x) for _ in range(2)]
    od = [torch.empty_like(out) for _ in range(2)]
    s_in, s_comp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()  # noqa: E731
    x_ready, comp_done, out_free = [ev(), ev()], [ev(), ev()], [ev(), ev()]
    x_free = [ev(), ev()]
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(s_comp)
    s_in.wait_event(t0)
    s_out.wait_event(t0)
    for i in range(n):
        b = i & 1
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(x_free[b])
            xd[b].copy_(xh, non_blocking=True)
            x_ready[b].record(s_in)
        with torch.cuda.stream(s_comp):
            s_comp.wait_event(x_ready[b])
            if i >= 2:
                s_comp.wait_event(out_free[b])
            step(xd[b], od[b])
            x_free[b].record(s_comp)
            comp_done[b].record(s_comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(comp_done[b])
            oh[b].copy_(od[b], non_blocking=True)
            out_free[b].record(s_out)
    s_comp.wait_stream(s_out)
    t1.record(s_comp)
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1)
    if pg:
        t = torch.tensor([ms], device=dev)
        pg.all_reduce(t, op=pg.ReduceOp.MAX)
        ms = t.item()
    world = pg.get_world_size() if pg else 1
    return {"value": world * p.T * n / (ms / 1000.0), "unit": "tokens/s",
            "h2d_bytes_per_step": xh.numel() * xh.element_size(),
            "d2h_bytes_per_step": oh[0].numel() * oh[0].element_size(), "steps": n,
            "path": "pinned host x -> moe_layer_forward (C ABI) -> pinned host out; copies of neighbouring "
                    "batches overlap the layer (3 streams, double buffers)"}


def run_standalone_memory_stages(B, cfg, p, x, w_router, bias, ws, f8, hbm, reps=20):
    """moe_route (router GEMM + selection), moe_permute and the routed sum of
    moe_combine timed on their own (CUDA events, main stream, nothing else
    running), with their algorithmic HBM bytes: the memory-bound part of the
    step without the side-stream overlap of the layer call. Inputs are the
    bench's; outputs go to buffers of their own."""
    dev = x.device
    T, E, K, d = p.T, p.E, p.K, p.d
    a_b = 2 if p.dtype == "bf16" else 4
    ex = 1 if f8 else a_b
    scores = torch.empty(T, E, device=dev)
    idx = torch.empty(T, K, dtype=torch.int32, device=dev)
    gate = torch.empty(T, K, device=dev)
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    off = torch.empty(E + 1, dtype=torch.int32, device=dev)
    st = torch.empty(T * K, dtype=torch.int32, device=dev)
    sp = torch.empty(T, K, dtype=torch.int32, device=dev)
    xp = torch.empty(T * K, d, dtype=torch.uint8 if f8 else x.dtype, device=dev)
    xs = torch.empty(d // 128, T * K, device=dev) if f8 else None
    b = bias.clone()

    def route():
        B.moe_route(cfg, x, w_router, None, b, scores, idx, gate, counts, ws)

    def permute():
        B.moe_permute(cfg, idx, counts, off, st, sp, x, xp, xs, ws)

    # the memory-bound part of the combine: the gate-weighted sum of each
    # token's K expert rows, which moe_combine runs alone for S = 0
    cfg0 = B.make_config(T, d, E, p.G, K, p.M, p.I, 0, p.group_topk, p.dtype, p.expert_dtype)
    yp = torch.zeros(T * K, d, dtype=x.dtype, device=dev)
    rsum = torch.empty(T, d, dtype=x.dtype, device=dev)
    no_w = B.make_weights()

    def combine():
        B.moe_combine(cfg0, yp, sp, gate, None, no_w, rsum, ws)

    out = {}
    route_bytes = T * d * a_b + E * d * a_b + 2 * T * E * 4 + T * K * 8
    perm_bytes = T * d * a_b + T * K * d * ex + T * K * 16 + (T * K * (d // 128) * 4 if f8 else 0)
    comb_bytes = T * K * d * a_b + T * d * a_b + T * K * 8
    for name, fn, nbytes in (("route", route, route_bytes), ("permute", permute, perm_bytes),
                             ("combine_routed_sum", combine, comb_bytes)):
        for _ in range(3):
            route()
            permute()
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / reps
        out[name] = {"ms": ms, "bytes": nbytes, "gbs": nbytes / (ms * 1e-3) / 1e9,
                     "frac_hbm": nbytes / (ms * 1e-3) / 1e9 / hbm}
    tot_b = route_bytes + perm_bytes
    tot_ms = out["route"]["ms"] + out["permute"]["ms"]
    out["route_permute"] = {"gbs": tot_b / (tot_ms * 1e-3) / 1e9, "frac_hbm": tot_b / (tot_ms * 1e-3) / 1e9 / hbm}
    tot_b += comb_bytes
    tot_ms += out["combine_routed_sum"]["ms"]
    out["route_permute_combine"] = {"gbs": tot_b / (tot_ms * 1e-3) / 1e9,
                                    "frac_hbm": tot_b / (tot_ms * 1e-3) / 1e9 / hbm}
    code = B.moe_device_error(ws)
    if code != 0:
        raise RuntimeError(f"device error 0x{code:x} in the standalone stages")
    return out


def layer_graphs_on():
    return os.environ.get("MOE_LAYER_GRAPHS", "1")[:1] != "0"


def run_graph_replay(step, p, K, dev, world):
    """One layer step captured into a CUDA graph (after the eager steps above
    created the library's side stream) and replayed K times, timed with CUDA
    events: the same kernels without per-launch host work."""
    if world != 1:
        return None
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    torch.cuda.synchronize()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(K):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / K
    return {"ms_per_step": ms, "value": p.T / (ms / 1000.0), "unit": "tokens/s", "steps": K,
            "note": "moe_layer_forward captured once into a CUDA graph and replayed"}


def kernels_per_step(p):
    """Kernels of this library one moe_layer_forward step launches (cudaMemset
    calls are not counted)."""
    f8 = p.expert_dtype in ("e4m3", "e4m3_ue8m0")
    scatter = p.combine == "scatter_add" and not f8
    n = 6  # router, selection, rank, scan, scatter, bias update
    n += 1  # routed GEMM1
    if p.S > 0:
        n += 1  # shared experts' GEMM1 (side stream)
    if scatter:
        n += 1 + (1 if p.S > 0 else 0)  # routed GEMM2 with the reductions; shared down projection (fp32 seed)
        n += 1 if p.dtype == "bf16" else 0  # rounding pass (fp32 layers add into out itself)
    else:
        n += 2 + (1 if p.S > 0 else 0)  # routed GEMM2, routed sum; shared down projection with the sum added
    if f8:
        n += 1 + (1 if p.S > 0 else 0)  # tile-major scale layout; x quantised for the shared experts
    if p.dtype == "f32":
        n += 4 + (2 if p.S > 0 else 0)  # x, router, routed and shared weights split into tf32 pairs
    return n


def load_slope(counts, top=16):
    """Log-log slope of the sorted expert loads over the top ranks against the
    rank of the skew direction (two experts share each of the 8 directions,
    so ranks 2j+1 and 2j+2 both have direction rank j+1)."""
    import numpy as np
    c = np.sort(np.asarray(counts, np.float64))[::-1][:top]
    r = np.arange(len(c), dtype=np.float64) // 2 + 1
    return float(np.polyfit(np.log(r), np.log(np.maximum(c, 1.0)), 1)[0])


def raw_routing_load(B, cfg, p, x, w_router, dev, ws):
    """The raw load of the workload: one moe_route with bias 0 on the bench's
    tokens, before any bias update."""
    counts = torch.empty(p.E, dtype=torch.int32, device=dev)
    idx = torch.empty(p.T, p.K, dtype=torch.int32, device=dev)
    gate = torch.empty(p.T, p.K, device=dev)
    B.moe_route(cfg, x, w_router, None, torch.zeros(p.E, device=dev), None, idx, gate, counts, ws)
    c = counts.cpu().double()
    return {"raw_load_max_over_mean": float(c.max() / c.mean()),
            "raw_load_loglog_slope_top16": load_slope(c.numpy()),
            "raw_load_note": "one routing of the bench tokens at bias 0, before warm-up; the slope is fitted "
                             "over the 16 hottest experts against their skew-direction rank"}


def run_cpu_baseline(p, w, x, min_seconds=10.0):
    """The C++ oracle unit (CpuOracleUnit) run back to back for about
    min_seconds, on the host cores, reported as the harmonic mean."""
    unit = CpuOracleUnit(p, w, x.cpu())
    vals, secs = [], 0.0
    while secs < min_seconds or len(vals) < 3:
        v, s = unit.run()
        vals.append(v)
        secs += s
    return {"value": len(vals) / sum(1.0 / v for v in vals), "unit": "tokens/s", "cores": CpuOracleUnit.cores(),
            "kind": "oracle", "sample": unit.desc + f" ({len(vals)} units)", "seconds": secs}


def time_layer(B, cfg, p, x, weights, bias, ws, dev, steps=20, warmup=3, stage_events=False):
    """moe_layer_forward with the workload's bias update, timed with CUDA
    events over `steps` steps after `warmup`; optional per-stage means."""
    out = torch.empty(p.T, p.d, dtype=synth.torch_dtype(p.dtype), device=dev)
    idx = torch.empty(p.T, p.K, dtype=torch.int32, device=dev)
    gate = torch.empty(p.T, p.K, dtype=torch.float32, device=dev)
    counts = torch.empty(p.E, dtype=torch.int32, device=dev)

    def step():
        B.moe_layer_forward(cfg, x, weights, bias, p.gamma, out, idx, gate, counts, None, ws)

    for _ in range(warmup):
        step()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(8)] for _ in range(steps)] if stage_events else None
    if ev:
        for row in ev:
            for e in row:
                e.record()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    for i in range(steps):
        if ev:
            B.moe_set_stage_events(ev[i])
        step()
    t1.record()
    torch.cuda.synchronize()
    if ev:
        B.moe_set_stage_events(None)
    code = B.moe_device_error(ws)
    if code != 0:
        raise RuntimeError(f"device error 0x{code:x} in {p.name}")
    ms = t0.elapsed_time(t1) / steps
    res = {"ms_per_step": ms, "tokens_per_s": p.T / (ms * 1e-3), "steps": steps, "counts": counts.cpu()}
    if ev:
        res["stage_ms"] = {name: sum(ev[i][j].elapsed_time(ev[i][j + 1]) for i in range(steps)) / steps
                           for j, name in enumerate(STAGES)}
    return res


def run_combine_ab(B, p, w, x, dev, rounds=3, steps=20):
    """Same-process A/B of the two combine modes on the headline workload:
    `rounds` alternations of `steps` timed steps each (after 3 warm-up
    steps), so that both see the same clock drift; the mean ms per step of
    each mode and the routed down projection + combine stages."""
    wd = {k: getattr(w, k).contiguous() for k in ("w_router", "w13", "w2", "ws13", "ws2")}
    res = {}
    for mode in ("gather", "scatter_add"):
        q = p.replace(combine=mode)
        cfg = B.config_from_preset(q)
        res[mode] = {"cfg": cfg, "ws": B.alloc_workspace(cfg, dev), "ms": [], "gemm2": [], "combine": []}
    for _ in range(rounds):
        for mode, r in res.items():
            q = p.replace(combine=mode)
            bias = synth.make_bias(q, device=dev)
            t = time_layer(B, r["cfg"], q, x, B.make_weights(**wd), bias, r["ws"], dev, steps=steps,
                           stage_events=True)
            r["ms"].append(t["ms_per_step"])
            r["gemm2"].append(t["stage_ms"]["gemm2_routed"])
            r["combine"].append(t["stage_ms"]["gemm2_shared_combine"])
    out = {}
    for mode, r in res.items():
        out[mode] = {"ms_per_step": sum(r["ms"]) / rounds, "ms_per_step_each": r["ms"],
                     "gemm2_routed_ms": sum(r["gemm2"]) / rounds, "combine_ms": sum(r["combine"]) / rounds}
        del r["ws"]
    torch.cuda.empty_cache()
    out["note"] = (f"{rounds} alternating rounds of {steps} steps per mode, same process, inputs and weights; "
                   "combine_ms is the stage after the routed down projection (gather: routed sum + shared down "
                   "projection; scatter_add: the fp32 -> bf16 rounding pass, the shared down projection runs on "
                   "the side stream)")
    return out


def run_other_workloads(B, w, dev, hbm, tf_sust):
    """The other configurations: the fp32 and mid-size parity layers (50
    steps each, weights of their own), the decode-shape batches (T = 64 and
    512) and the FP8 workload (T = 32768, fp32 and power-of-two tile scales),
    each timed the same way as the headline (20 steps) on the V3 weights
    already on the device (the decode shapes share them; the FP8 workloads
    quantise them)."""
    out = {}
    # the parity-size configurations, each with weights of its own shape
    for name in ("tiny_t256_d512_e16_fp32", "mid_t4096_d2048_e64_bf16"):
        q = synth.PRESETS[name]
        wq = synth.make_weights(q, device=dev)
        cfg = B.config_from_preset(q)
        ws = B.alloc_workspace(cfg, dev)
        x = synth.make_x(q, wq.w_router, device=dev)
        bias = synth.make_bias(q, device=dev)
        W = B.make_weights(**{k: getattr(wq, k).contiguous() for k in ("w_router", "w13", "w2", "ws13", "ws2")})
        r = time_layer(B, cfg, q, x, W, bias, ws, dev, steps=50, stage_events=True)
        fl = flops_gemm1(q) + flops_gemm2_routed(q)
        g_ms = r["stage_ms"]["gemm1_swiglu"] + r["stage_ms"]["gemm2_routed"]
        out[name] = {"ms_per_step": r["ms_per_step"], "tokens_per_s": r["tokens_per_s"],
                     "expert_gemm_tflops": fl / (g_ms * 1e-3) / 1e12,
                     "note": "fp32 operands as tf32 pairs (three MMAs per product)" if q.dtype == "f32" else "bf16"}
        del ws, x, wq, W
    torch.cuda.empty_cache()
    wd = {k: getattr(w, k).contiguous() for k in ("w_router", "w13", "w2", "ws13", "ws2")}
    for name in ("v3_decode_t64_bf16", "v3_decode_t512_bf16"):
        q = synth.PRESETS[name]
        cfg = B.config_from_preset(q)
        ws = B.alloc_workspace(cfg, dev)
        x = synth.make_x(q, w.w_router, device=dev)
        bias = synth.make_bias(q, device=dev)
        r = time_layer(B, cfg, q, x, B.make_weights(**wd), bias, ws, dev)
        hit = int((r["counts"] > 0).sum())
        nbytes = (hit + q.S) * 3 * q.d * q.I * 2
        out[name] = {"ms_per_step": r["ms_per_step"], "tokens_per_s": r["tokens_per_s"], "experts_hit": hit,
                     "weight_bytes": nbytes, "gbs": nbytes / (r["ms_per_step"] * 1e-3) / 1e9,
                     "frac_hbm": nbytes / (r["ms_per_step"] * 1e-3) / 1e9 / hbm}
        del ws, x
    for name in ("v3_t32768_d7168_e256_fp8", "v3_t32768_d7168_e256_fp8_ue8m0"):
        q = synth.PRESETS[name]
        quant = B.moe_quantize_weights_e4m3_ue8m0 if q.expert_dtype == "e4m3_ue8m0" else B.moe_quantize_weights_e4m3
        wq = {"w_router": wd["w_router"]}
        for k in ("w13", "w2", "ws13", "ws2"):
            m = wd[k]
            qt = torch.empty(m.shape, dtype=torch.uint8, device=dev)
            sc = torch.empty((m.shape[0], (m.shape[1] + 127) // 128, (m.shape[2] + 127) // 128),
                             dtype=torch.float32, device=dev)
            quant(m, qt, sc)
            wq[k], wq[k + "_scale"] = qt, sc
        cfg = B.config_from_preset(q)
        ws = B.alloc_workspace(cfg, dev)
        x = synth.make_x(q, w.w_router, device=dev)
        bias = synth.make_bias(q, device=dev)
        r = time_layer(B, cfg, q, x, B.make_weights(**wq), bias, ws, dev, stage_events=True)
        g1 = flops_gemm1(q) / (r["stage_ms"]["gemm1_swiglu"] * 1e-3) / 1e12
        out[name] = {"ms_per_step": r["ms_per_step"], "tokens_per_s": r["tokens_per_s"],
                     "gemm1_ms": r["stage_ms"]["gemm1_swiglu"], "gemm1_tflops": g1,
                     "gemm1_frac_fp8_sustained": g1 / (2 * tf_sust),
                     "gemm2_routed_ms": r["stage_ms"]["gemm2_routed"]}
        del ws, x, wq
        torch.cuda.empty_cache()
    out["note"] = ("same process and box as the headline, 20 timed steps (50 for the parity-size layers) after 3 "
                   "warm-up steps each (forward + bias update); FP8 peak = 2 x the measured bf16 sustained peak "
                   "(nominal fp8 / bf16 ratio)")
    return out


# ---------------------------------------------------------------- our arm
def run_ours(a, p):
    from mixture_experts_layer_100_b300 import binding as B
    from mixture_experts_layer_100_b300 import dp

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist
    # replicas: same weights on every rank, an independent token batch per rank
    w = synth.make_weights(p, device=dev)
    x = synth.make_x(p.replace(seed=p.seed + rank) if rank else p, w.w_router, device=dev)
    bias = synth.make_bias(p, device=dev)
    cfg = B.config_from_preset(p)
    ws = B.alloc_workspace(cfg, dev)
    wd = {k: getattr(w, k).contiguous() for k in ("w_router", "w13", "w2", "ws13", "ws2")}
    f8 = p.expert_dtype in ("e4m3", "e4m3_ue8m0")
    if f8:
        # expert weights to e4m3 with 128x128 block scales, once, before timing
        quant = B.moe_quantize_weights_e4m3_ue8m0 if p.expert_dtype == "e4m3_ue8m0" else B.moe_quantize_weights_e4m3
        for k in ("w13", "w2", "ws13", "ws2"):
            m = wd[k]
            q = torch.empty(m.shape, dtype=torch.uint8, device=dev)
            sc = torch.empty((m.shape[0], (m.shape[1] + 127) // 128, (m.shape[2] + 127) // 128),
                             dtype=torch.float32, device=dev)
            quant(m, q, sc)
            wd[k], wd[k + "_scale"] = q, sc
        torch.cuda.synchronize()
    weights = B.make_weights(**wd)
    out = torch.empty(p.T, p.d, dtype=synth.torch_dtype(p.dtype), device=dev)
    idx = torch.empty(p.T, p.K, dtype=torch.int32, device=dev)
    gate = torch.empty(p.T, p.K, dtype=torch.float32, device=dev)
    counts = torch.empty(p.E, dtype=torch.int32, device=dev)
    mom = torch.empty(1, dtype=torch.float32, device=dev)
    gamma = p.gamma

    update = dp.device_bias_update(cfg, gamma, bias, mom)

    def step(xin=None, o=None):
        xin = x if xin is None else xin
        o = out if o is None else o
        if world == 1:
            B.moe_layer_forward(cfg, xin, weights, bias, gamma, o, idx, gate, counts, mom, ws)
        else:
            # the bias sees the load of the whole data-parallel batch: counts
            # are summed over ranks (1 KB all-reduce) before the update
            B.moe_layer_forward(cfg, xin, weights, bias, 0.0, o, idx, gate, counts, mom, ws)
            dp.global_bias_update(counts, p.T, update)

    raw_load = raw_routing_load(B, cfg, p, x, wd["w_router"], dev, ws)
    for _ in range(a.warmup):
        step()
    torch.cuda.synchronize()
    code = B.moe_device_error(ws)
    if code != 0:
        raise RuntimeError(f"device error 0x{code:x} during warm-up")

    K = a.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(8)] for _ in range(K)]
    for row in ev:  # create the event objects before handing them to the library
        for e in row:
            e.record()
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    if pg:
        pg.barrier()
    sampler = ClockSampler(local, enabled=not a.no_clocks and rank == 0)
    with sampler:
        torch.cuda.synchronize()
        sampler.mark_start()
        t_start.record()
        for i in range(K):
            B.moe_set_stage_events(ev[i])
            step()
        t_end.record()
        torch.cuda.synchronize()
        sampler.mark_end()
    B.moe_set_stage_events(None)
    if pg:
        pg.barrier()
    ms = t_start.elapsed_time(t_end)
    if pg:
        t = torch.tensor([ms], device=dev)
        pg.all_reduce(t, op=pg.ReduceOp.MAX)
        ms = t.item()
    code = B.moe_device_error(ws)
    if code != 0:
        raise RuntimeError(f"device error 0x{code:x} in the timed region")
    value = world * p.T * K / (ms / 1000.0)
    stage_ms = {name: sum(ev[i][j].elapsed_time(ev[i][j + 1]) for i in range(K)) / K
                for j, name in enumerate(STAGES)}

    hbm, tf_burst, tf_sust, src = peaks()
    if f8:
        # FP8 dense peak: the measured bf16 peak times the nominal fp8 / bf16 ratio (4.5 / 2.25)
        tf_burst, tf_sust, src = 2 * tf_burst, 2 * tf_sust, src + " bf16 x 2 (nominal fp8 ratio)"
    g1 = flops_gemm1(p) / (stage_ms["gemm1_swiglu"] * 1e-3) / 1e12
    roofline = {"kernel": "gemm1_swiglu (routed experts, tcgen05)", "bound": "tensor",
                "achieved": g1, "peak": tf_sust, "unit": "TFLOP/s", "frac": g1 / tf_sust,
                "peak_kind": f"{'fp8' if f8 else 'bf16'} dense, sustained ({src})",
                "frac_of_burst_peak": g1 / tf_burst,
                "traffic": traffic_from_profiles("gemm1_swiglu", p.expert_dtype)}
    stages = {}
    hb = hbm_bytes(p)
    for name in STAGES:
        st = {"ms": stage_ms[name]}
        if name in ("gemm1_swiglu", "gemm2_routed", "gemm2_shared_combine"):
            fl = {"gemm1_swiglu": flops_gemm1, "gemm2_routed": flops_gemm2_routed,
                  "gemm2_shared_combine": flops_gemm2_shared}[name](p)
            st["tflops"] = fl / (stage_ms[name] * 1e-3) / 1e12
            st["frac_tensor_sustained"] = st["tflops"] / tf_sust
        if name in hb:
            st["gbs"] = hb[name] / (stage_ms[name] * 1e-3) / 1e9
            st["frac_hbm"] = st["gbs"] / hbm
        stages[name] = st
    gemm_ms = stage_ms["gemm1_swiglu"] + stage_ms["gemm2_routed"]
    expert_gemm_tf = (flops_gemm1(p) + flops_gemm2_routed(p)) / (gemm_ms * 1e-3) / 1e12
    mem_ms = stage_ms["router_gemm"] + stage_ms["route_select"] + stage_ms["permute"]
    mem_gbs = (hb["router_gemm"] + hb["route_select"] + hb["permute"]) / (mem_ms * 1e-3) / 1e9

    # sequence-wise balance statistic of the last step's routing (runs of
    # 4096 tokens; alpha 1, so the value is sum_i f_i P_i itself)
    seq_len = min(4096, p.T)
    n_seq = (p.T + seq_len - 1) // seq_len
    sb_loss = torch.empty(n_seq, device=dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    B.moe_seq_balance(cfg, None, idx, seq_len, 1.0, sb_loss, None, None, ws)
    e1.record()
    torch.cuda.synchronize()
    seq_balance = {"seq_len": seq_len, "alpha": 1.0, "per_sequence": [round(v, 6) for v in sb_loss.tolist()],
                   "ms": e0.elapsed_time(e1),
                   "note": "moe_seq_balance on the last step's affinities and choices; 1.0 = perfectly even"}

    graph = None
    if not a.no_graph:
        graph = run_graph_replay(step, p, K, dev, world)
        code = B.moe_device_error(ws)
        if code != 0:
            raise RuntimeError(f"device error 0x{code:x} in the graph replay")

    standalone = None
    if rank == 0 and not a.no_standalone:
        standalone = run_standalone_memory_stages(B, cfg, p, x, wd["w_router"], bias, ws, f8, hbm)

    e2e = None
    if not a.no_e2e:
        e2e = run_e2e(a, p, x, out, step, dev, pg)

    cpu = None
    if rank == 0 and world == 1 and not a.no_cpu_baseline:
        cpu = run_cpu_baseline(p, w, x)

    extra = None
    if rank == 0 and world == 1 and not a.no_extra and p == synth.PRESETS[DEFAULT_PRESET]:
        # only for the unmodified headline workload: the other configurations reuse its V3 weights
        del ws
        torch.cuda.empty_cache()
        extra = {"combine_ab": run_combine_ab(B, p, w, x, dev)}
        extra.update(run_other_workloads(B, w, dev, hbm, tf_sust))

    clocks = sampler.summary() if rank == 0 else None
    if rank == 0:
        cfg_line = bench_config(p, world)
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K,
            "warmup": a.warmup, "ms_per_step": ms / K, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16" if p.expert_dtype == "bf16" else p.expert_dtype,
            "data": "synthetic (seeded; random-init weights N(0, 0.006); x ~ N(0,1) + rank-8 routing skew)",
            "config": cfg_line,
            "raw_routing_load": raw_load,
            "roofline": roofline,
            "stages": stages,
            "expert_gemms": {"tflops": expert_gemm_tf, "frac_tensor_sustained": expert_gemm_tf / tf_sust,
                             "frac_tensor_burst": expert_gemm_tf / tf_burst},
            "route_permute_hbm": {"gbs": mem_gbs, "frac_hbm": mem_gbs / hbm,
                                  "note": "stage times inside the step, where the shared experts' GEMM1 runs "
                                          "beside routing and permutation on a side stream"},
            "memory_stages_standalone": standalone,
            "graph_replay": graph,
            "seq_balance": seq_balance,
            "cpu_baseline": cpu,
            "other_workloads": extra,
            "e2e": e2e,
            "gpu_launches": kernels_per_step(p) * K,
            "launch": {"layer_graphs": layer_graphs_on(),
                       "note": "moe_layer_forward replays a CUDA graph of its kernels, captured by the library at "
                               "the second call with the same arguments (MOE_LAYER_GRAPHS=0 launches them one "
                               "by one); gpu_launches counts the kernels either way"},
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    if pg:
        pg.barrier()
        pg.destroy_process_group()


def main():
    a = parse()
    p = preset_from_args(a)
    if a.impl == "reference":
        run_reference(a, p)
    else:
        run_ours(a, p)


if __name__ == "__main__":
    main()
