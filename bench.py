"""Benchmark of the fused MoE router on GB300.

Headline workload (one "step"): the decode router at M=8 verify rows,
H=2048, E=256, top-8 softmax, run for 40 MoE layers back to back, each
layer with its own W_gate, captured once as a CUDA graph and replayed. The
W_gate pool rotates over 520 MiB (> the 129 MB L2), so every call streams
its weights from HBM. Value = router tokens/s = rows routed per second
summed over the layer calls (M x 40 per step).

Also reported (``detail``): per-call latency and roofline fraction at each
configuration of the router pages (decode M=1/2/8, sqrt-softplus+bias
M=1/16/64, the M=16384 prefill with BF16 and NVFP4 weights, and the M=2
router with its unique-route table), the fused-versus-unfused A/B, and the
CPU oracle's throughput.

``--impl reference`` times the CPU oracle on the same workload instead.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

LAYERS = 40          # router calls per decode token (one per MoE layer)

# DRAM bytes per launch of the headline kernel from one ncu capture of the
# decode workload, valid only for the sources that kernel is built from: its
# file (kernel and launcher) and the headers that file includes.
DECODE_SOURCES = ("gemv.cu", "kernels.h", "select.cuh", "dfkey.cuh", "common.cuh")
TRAFFIC = {"decode": {"bytes": 1156693, "src_sha": "b0cadfb85b80161a"}}


def kernel_src_sha(files=DECODE_SOURCES):
    import hashlib
    h = hashlib.sha256()
    for f in sorted(files):
        h.update(f.encode())
        with open(os.path.join(ROOT, "moe_expert_router_02_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def traffic_for(name):
    t = TRAFFIC.get(name)
    return t["bytes"] if t and t["src_sha"] == kernel_src_sha() else None


W_POOL_BYTES = 520 << 20


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return dict(hbm=float(p["hbm_gbs"]), bf16=float(p["bf16_tflops"]),
                    bf16_sus=float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                    source="measured")
    except Exception:
        return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, source="fallback")


class Clocks:
    """nvidia-smi sampling during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu: int):
        self.gpu = gpu
        self.p = None

    def __enter__(self):
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                                       "--format=csv,noheader,nounits", "-lms", "200"],
                                      stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.p = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.p is not None:
            time.sleep(0.25)
            self.p.terminate()
            try:
                out, _ = self.p.communicate(timeout=5)
                self.lines = [l for l in out.splitlines() if l.strip()]
            except Exception:
                self.p.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup(n_gpus):
    rank, world = int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v, world):
    """Largest value over all ranks (the job's time is its slowest rank's)."""
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    device = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(rows_per_rank, layers, steps, world, ms_max):
    """Whole-job router tokens/s: every rank routes its own batch (replicas,
    no exchange), and the job takes as long as its slowest rank."""
    return rows_per_rank * layers * steps * world / (ms_max / 1e3)


# ---------------------------------------------------------------- GPU helpers
def dev(a):
    import torch
    a = np.ascontiguousarray(a)
    return torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).cuda()


def time_graph(graph_fn, reps, warm=3):
    """Average ms of graph_fn() over reps, CUDA events on the current stream."""
    import torch
    for _ in range(warm):
        graph_fn()
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record()
    for _ in range(reps):
        graph_fn()
    e.record()
    torch.cuda.synchronize()
    return s.elapsed_time(e) / reps


class RouterSet:
    """A pool of distinct (x, W) inputs for one configuration, with graphs
    of ``calls`` back-to-back router calls over consecutive pool slots."""

    def __init__(self, cfg, M, calls, w_dtype=None, pool_bytes=W_POOL_BYTES, table=False,
                 flags=0, seed=0):
        import torch

        from moe_expert_router_02_gb300 import router as R
        from moe_expert_router_02_gb300 import synth
        self.R, self.cfg, self.M, self.calls, self.table = R, cfg, M, calls, table
        self.H, self.E, self.k, self.act = cfg["H"], cfg["E"], cfg["k"], cfg["act"]
        case = synth.make_case(cfg, M=M, seed=seed, w_dtype=w_dtype)
        self.case = case
        wb = case["W"].nbytes + (0 if case["scales"] is None else case["scales"].nbytes)
        self.w_bytes = wb
        n_w = max(calls, int(np.ceil(pool_bytes / wb)))
        n_w = int(np.ceil(n_w / calls) * calls)
        self.n_graphs = n_w // calls
        W0 = dev(case["W"])
        self.W = W0.unsqueeze(0).repeat(n_w, *([1] * W0.dim()))  # distinct buffers, same values
        self.scales = None if case["scales"] is None else dev(case["scales"])
        self.x = dev(case["x"]).unsqueeze(0).repeat(calls, *([1] * 2)).contiguous()
        self.bias = None if case["bias"] is None else dev(case["bias"])
        self.idx = torch.empty((calls, M, self.k), dtype=torch.int32, device="cuda")
        self.w = torch.empty((calls, M, self.k), dtype=torch.float32, device="cuda")
        self.tbl = None
        if table:
            n = 2 * self.k
            G = M // 2
            self.tbl = (torch.empty((calls, G, n), dtype=torch.int32, device="cuda"),
                        torch.empty((calls, G, n), dtype=torch.uint8, device="cuda"),
                        torch.empty((calls, G, 2, self.k), dtype=torch.uint8, device="cuda"),
                        torch.empty((calls, G), dtype=torch.int32, device="cuda"))
        self.flags = flags
        self.stream = torch.cuda.Stream()
        self.graphs = []

    def opts(self, c):
        tbl = None if self.tbl is None else tuple(t[c] for t in self.tbl)
        return self.R.make_opts(x_dtype=self.case["x_dtype"], w_dtype=self.case["w_dtype"],
                                w_scales=self.scales, w_global_scale=self.case["g"], table=tbl,
                                flags=self.flags)

    def call(self, c, wslot, stream):
        self.R.router_forward_ex(self.x[c], self.W[wslot], self.bias, self.M, self.H, self.E,
                                 self.k, self.act, self.idx[c], self.w[c], self.opts(c),
                                 stream=stream)

    def capture(self):
        import torch
        s = self.stream
        with torch.cuda.stream(s):
            for c in range(self.calls):  # sizes the library workspace outside capture
                self.call(c, c, s)
        s.synchronize()
        for gi in range(self.n_graphs):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                for c in range(self.calls):
                    self.call(c, gi * self.calls + c, s)
            self.graphs.append(g)
        torch.cuda.synchronize()
        self.step_i = 0

    def step(self):
        self.graphs[self.step_i % self.n_graphs].replay()
        self.step_i += 1

    def algo_bytes(self):
        M, H, E, k = self.M, self.H, self.E, self.k
        xb = M * H * (4 if self.case["x_dtype"] == 0 else 2)
        out = M * k * 8 + (0 if self.case["bias"] is None else E * 4)
        tbl = 0 if not self.table else (M // 2) * (2 * k * 4 + 2 * k + 2 * k + 4)
        return self.w_bytes + xb + out + tbl


def per_call_stats(rs, steps):
    """(us per call in the back-to-back graph, us of one call alone).

    The single call is a one-kernel CUDA graph replayed with the device idle
    before it, so the figure includes the graph launch but no host Python."""
    import torch
    ms = time_graph(rs.step, steps)
    us_pipe = ms * 1e3 / rs.calls
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=rs.stream):
        rs.call(0, 0, rs.stream)
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    tot = 0.0
    n = 30
    for i in range(n + 3):
        torch.cuda.synchronize()
        s.record()
        g.replay()
        e.record()
        torch.cuda.synchronize()
        if i >= 3:
            tot += s.elapsed_time(e)
    return us_pipe, tot * 1e3 / n


# ---------------------------------------------------------------- CPU oracle timing
def oracle_tokens_per_s(cfg, M, budget_s=10.0, min_calls=1, w_dtype=None, rows=None):
    """Oracle router throughput on host cores (single thread)."""
    import oracle
    from moe_expert_router_02_gb300 import synth
    case = synth.make_case(cfg, M=M, seed=0, w_dtype=w_dtype)
    if rows is not None:  # bounded sample of a large batch
        case = dict(case, M=rows, x=case["x"][:rows])
    t0 = time.perf_counter()
    calls = 0
    while calls < min_calls or time.perf_counter() - t0 < budget_s:
        oracle.router(case)
        calls += 1
    dt = time.perf_counter() - t0
    return case["M"] * calls / dt, calls, dt


def host_cores():
    """Cores this process may run on (its affinity set)."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_prefill(cfg, budget_s=10.0):
    """The oracle on the prefill workload (M=16384, H=7168, E=256, k=8,
    sqrt-softplus + bias, BF16): 256 rows on one core, and row slices on
    every core of the affinity set at once (threads: the oracle's C code
    runs without the interpreter lock), each extrapolated to all 16384 rows.
    The oracle's arithmetic is untouched; only its rows are split."""
    import concurrent.futures as cf

    import oracle
    from moe_expert_router_02_gb300 import synth
    case = synth.make_case(cfg, seed=0)
    M = case["M"]

    def rows(a, b):
        return dict(case, M=b - a, x=case["x"][a:b])

    t0 = time.perf_counter()
    oracle.router(rows(0, 256))
    one = time.perf_counter() - t0
    cores = host_cores()
    # as many rows per core as one core did in about budget_s / 2 seconds
    per = max(16, min(M // cores, int(256 * (budget_s / 2) / max(one, 1e-3))))
    t0 = time.perf_counter()
    with cf.ThreadPoolExecutor(max_workers=cores) as ex:
        list(ex.map(lambda c: oracle.router(rows(c * per, (c + 1) * per)), range(cores)))
    par = time.perf_counter() - t0
    return {"unit": "router tokens/s", "single_core": 256 / one,
            "single_core_call_s_extrapolated": one * M / 256,
            "all_cores": cores * per / par, "all_cores_call_s_extrapolated": par * M / (cores * per),
            "cores": cores,
            "sample": f"256 rows on one core ({one:.1f} s); {per} rows on each of {cores} cores "
                      f"at once ({par:.1f} s)"}


# ---------------------------------------------------------------- main arms
def run_ours(args, rank, world, local):
    import torch

    from moe_expert_router_02_gb300 import router as R
    from moe_expert_router_02_gb300 import synth
    torch.cuda.set_device(local)
    peaks = load_peaks()
    C = synth.CONFIGS
    M = 8
    head = RouterSet(C["C1"], M, LAYERS)
    head.capture()
    for _ in range(args.warmup):
        head.step()
    torch.cuda.synchronize()
    barrier(world)
    ev_s, ev_e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with Clocks(local) as clk:
        torch.cuda.synchronize()
        ev_s.record()
        for _ in range(args.steps):
            head.step()
        ev_e.record()
        torch.cuda.synchronize()
    barrier(world)
    ms = ev_s.elapsed_time(ev_e)
    ms = max_over_ranks(ms, world)
    tokens = M * LAYERS * args.steps * world
    value = job_throughput(M, LAYERS, args.steps, world, ms)
    us_call = ms * 1e3 / (args.steps * LAYERS)
    algo = head.algo_bytes()
    achieved = algo / (us_call * 1e-6) / 1e9

    # end to end through the public API with host buffers: the 40 layer calls
    # are router_forward calls captured once as a CUDA graph (how a decode
    # loop issues them); every step copies its x from pinned host memory,
    # replays the calls and copies the ids and weights back
    x_host = torch.empty((LAYERS, M, head.H), dtype=torch.int16).pin_memory()
    x_host.copy_(head.x.cpu())
    idx_host = torch.empty((LAYERS, M, head.k), dtype=torch.int32).pin_memory()
    w_host = torch.empty((LAYERS, M, head.k), dtype=torch.float32).pin_memory()
    s = head.stream
    n_w = head.W.shape[0]
    with torch.cuda.stream(s):
        for c in range(LAYERS):  # the library workspace exists before capture
            R.router_forward(head.x[c], head.W[c], None, M, head.H, head.E, head.k, head.act,
                             head.idx[c], head.w[c], stream=s)
    s.synchronize()
    e2e_graphs = []
    for gi in range(head.n_graphs):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for c in range(LAYERS):
                R.router_forward(head.x[c], head.W[(gi * LAYERS + c) % n_w], None, M, head.H,
                                 head.E, head.k, head.act, head.idx[c], head.w[c], stream=s)
        e2e_graphs.append(g)

    def e2e_step(i):
        head.x.copy_(x_host, non_blocking=True)
        e2e_graphs[i % len(e2e_graphs)].replay()
        idx_host.copy_(head.idx, non_blocking=True)
        w_host.copy_(head.w, non_blocking=True)

    with torch.cuda.stream(s):
        for i in range(args.warmup):
            e2e_step(i)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for i in range(args.steps):
            e2e_step(i)
        torch.cuda.synchronize()
        e2e_s = time.perf_counter() - t0
    e2e_value = max_over_ranks(e2e_s, world)
    e2e_value = tokens / e2e_value
    del e2e_graphs

    detail = {}
    if not args.quick and rank == 0:
        detail = run_detail(args, peaks)

    cpu = None
    if rank == 0 and world == 1:
        tps, calls, dt = oracle_tokens_per_s(C["C1"], M, budget_s=args.cpu_budget)
        cpu = {"value": tps, "unit": "router tokens/s", "cores": 1, "kind": "oracle",
               "sample": f"{calls} oracle router calls at M=8, H=2048, E=256, k=8 "
                         f"({dt:.1f} s, single thread)",
               "host_cores": host_cores()}
        if not args.quick:
            cpu["prefill"] = oracle_prefill(C["C3"], args.cpu_budget)

    line = {
        "metric": "router tokens/s (decode M=8, H=2048, E=256, top-8 softmax, 40 layers)",
        "value": value, "unit": "router tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "decode router: M=8 rows, H=2048, E=256, k=8, softmax, "
                               "BF16 x (RMS-normalised rows) and W_gate ~ N(0,0.02), "
                               "40 layer calls per step (one CUDA graph)",
                   "l2": "W_gate pool of 520 MiB rotated (> 129 MB L2)",
                   "parallelism": f"replicas x{world}"},
        "us_per_call": us_call,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm"], "unit": "GB/s",
                     "frac": achieved / peaks["hbm"], "traffic": traffic_for("decode"),
                     "algo_bytes_per_call": algo, "peak_source": peaks["source"]},
        "e2e": {"value": e2e_value, "unit": "router tokens/s",
                "h2d_bytes_per_step": int(x_host.numel() * 2),
                "d2h_bytes_per_step": int(idx_host.numel() * 4 + w_host.numel() * 4)},
        "gpu_launches": args.steps * LAYERS,
        "clocks": clk.summary(),
        "cpu_baseline": cpu,
        "detail": detail,
    }
    if rank == 0:
        print(json.dumps(line))


def run_detail(args, peaks):
    """Per-configuration latency and roofline figures."""
    import torch

    from moe_expert_router_02_gb300 import router as R
    from moe_expert_router_02_gb300 import synth
    C = synth.CONFIGS
    out = {}

    def record(name, rs, steps=20, flops=None):
        rs.capture()
        us_pipe, us_iso = per_call_stats(rs, steps)
        algo = rs.algo_bytes()
        ent = {"M": rs.M, "us_per_call_pipelined": us_pipe, "us_per_call_isolated": us_iso,
               "tokens_per_s": rs.M / (us_pipe * 1e-6),
               "hbm_frac_pipelined": algo / (us_pipe * 1e-6) / 1e9 / peaks["hbm"],
               "hbm_frac_isolated": algo / (us_iso * 1e-6) / 1e9 / peaks["hbm"],
               "algo_bytes": algo,
               "regime": R.router_regime(rs.M, rs.H, rs.E, rs.k, rs.opts(0))}
        if flops:
            ent["tflops"] = flops / (us_pipe * 1e-6) / 1e12
            ent["bf16_frac"] = ent["tflops"] / peaks["bf16"]
        out[name] = ent
        del rs
        torch.cuda.empty_cache()

    for M in (1, 2, 8):
        record(f"C1_softmax_M{M}", RouterSet(C["C1"], M, LAYERS))
    # floors of a dependent call with the single-cluster kernel's launch shape
    # (include/gbrouter_diag.h): a chain of launches that only release and
    # wait, and one that also reads the call's x (8 x 2048 BF16)
    try:
        xs = torch.zeros((8, C["C1"]["H"]), dtype=torch.int16, device="cuda")
        sink = torch.zeros(16, dtype=torch.int32, device="cuda")
        fs = torch.cuda.Stream()
        for kind, name in ((0, "C1_floor_pdl_chain"), (1, "C1_floor_pdl_chain_read_x")):
            with torch.cuda.stream(fs):
                R.diag_chain(kind, LAYERS, xs, sink, fs)
            fs.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=fs):
                R.diag_chain(kind, LAYERS, xs, sink, fs)
            out[name] = {"us_per_launch": time_graph(g.replay, 20) * 1e3 / LAYERS}
        if "C1_softmax_M8" in out:
            out["C1_M8_us_above_read_x_floor"] = (out["C1_softmax_M8"]["us_per_call_pipelined"] -
                                                 out["C1_floor_pdl_chain_read_x"]["us_per_launch"])
    except Exception as e:  # a detail row never costs the headline line
        out["C1_floor"] = {"error": str(e)[:200]}
    record("C1_softmax_M8_unfused", RouterSet(C["C1"], 8, LAYERS, flags=R.GBR_FLAG_UNFUSED))
    for M in (1, 16, 64):
        record(f"C2_sqrtsoftplus_bias_M{M}", RouterSet(C["C2"], M, LAYERS))
    for M in (1, 16):  # the same router with NVFP4 W_gate (decoded in the kernel)
        record(f"C2_sqrtsoftplus_bias_M{M}_nvfp4",
               RouterSet(C["C2"], M, LAYERS, w_dtype=synth.NVFP4))
    for M in (1, 16):  # the sigmoid score with the same selection bias
        record(f"C2_sigmoid_bias_M{M}", RouterSet(dict(C["C2"], act=synth.SIGMOID), M, LAYERS))
    record("C4_M2_router_table", RouterSet(C["C4"], 2, LAYERS, table=True))
    record("C4_M2_router_no_table", RouterSet(C["C4"], 2, LAYERS))
    if "C4_M2_router_table" in out:
        out["C4_table_overhead_us"] = (out["C4_M2_router_table"]["us_per_call_pipelined"] -
                                       out["C4_M2_router_no_table"]["us_per_call_pipelined"])
    # unique-route table alone over 1e5 groups: a CUDA graph of back-to-back
    # calls over 12 distinct input/output sets (149 MB, more than L2), so
    # each call reads its ids from HBM and the host's launch rate is not timed
    G, k = C["C4"]["table_groups"], C["C4"]["k"]
    nset = 12
    idx = dev(synth.table_pairs(G, k, 256, seed=0))
    sets = []
    for _ in range(nset):
        sets.append((idx.clone(), torch.empty((G, 2 * k), dtype=torch.int32, device="cuda"),
                     torch.empty((G, 2 * k), dtype=torch.uint8, device="cuda"),
                     torch.empty((G, 2, k), dtype=torch.uint8, device="cuda"),
                     torch.empty((G,), dtype=torch.int32, device="cuda")))
    ts = torch.cuda.Stream()
    with torch.cuda.stream(ts):
        for st_ in sets:
            R.route_table(st_[0], G, 2, k, *st_[1:], stream=ts)
    ts.synchronize()
    tg = torch.cuda.CUDAGraph()
    with torch.cuda.graph(tg, stream=ts):
        for st_ in sets:
            R.route_table(st_[0], G, 2, k, *st_[1:], stream=ts)
    ms = time_graph(tg.replay, 10) / nset
    tbytes = G * (2 * k * 4 + 2 * k * 4 + 2 * k + 2 * k + 4)
    out["C4_table_only_1e5"] = {"us": ms * 1e3, "hbm_frac": tbytes / (ms * 1e-3) / 1e9 / peaks["hbm"],
                                "algo_bytes": tbytes, "timing": f"graph of {nset} calls on distinct sets"}
    del sets, tg
    torch.cuda.empty_cache()
    # the table's consumer: routed gather + shared-expert add over 10^3 groups
    # (M=2, k=6, D=4096 BF16 rows; 131 MB of rows, more than L2)
    Gg, kg, Dg = 1000, C["C4"]["k"], C["C4"]["H"]
    yg, wg, sg = synth.gather_inputs(Gg, kg, Dg, seed=0)
    tg = (torch.empty((Gg, 2 * kg), dtype=torch.int32, device="cuda"),
          torch.empty((Gg, 2 * kg), dtype=torch.uint8, device="cuda"),
          torch.empty((Gg, 2, kg), dtype=torch.uint8, device="cuda"),
          torch.empty((Gg,), dtype=torch.int32, device="cuda"))
    R.route_table(dev(synth.table_pairs(Gg, kg, 256, seed=1)), Gg, 2, kg, *tg)
    md = tg[2]
    mpg = md.cpu().numpy()
    yd, wd_, sd = dev(yg.view(np.int16)), dev(wg), dev(sg.view(np.int16))
    od = torch.empty((Gg, 2, Dg), dtype=torch.int16, device="cuda")
    ms = time_graph(lambda: R.route_gather_add(yd, md, wd_, sd, Gg, 2, kg, Dg, od), 20)
    rows_read = int(sum(len(set(mpg[g, t])) for g in range(Gg) for t in range(2)))
    gbytes = rows_read * Dg * 2 + 2 * (Gg * 2 * Dg * 2) + Gg * 2 * kg * 5
    out["C4_gather_add_1e3"] = {"us": ms * 1e3, "hbm_frac": gbytes / (ms * 1e-3) / 1e9 / peaks["hbm"],
                                "algo_bytes": gbytes}
    del yd, od
    torch.cuda.empty_cache()
    # prefill
    cfg3 = C["C3"]
    flops = 2 * cfg3["M"] * cfg3["H"] * cfg3["E"]
    for name, wd, act in (("C3_prefill_bf16", synth.BF16, cfg3["act"]),
                          ("C3_prefill_nvfp4", synth.NVFP4, cfg3["act"]),
                          ("C3_prefill_bf16_sigmoid", synth.BF16, synth.SIGMOID)):
        rs = RouterSet(dict(cfg3, act=act), cfg3["M"], 1, w_dtype=wd, pool_bytes=0)
        record(name, rs, steps=10, flops=flops)
    # smaller prefill batches of the same shape: stream-K spreads their few
    # tiles over more SMs (router_tc_groups pairs)
    for M in (4096, 8192):
        name = f"C3_prefill_bf16_M{M}"
        try:
            record(name, RouterSet(cfg3, M, 1, pool_bytes=0), steps=10,
                   flops=2 * M * cfg3["H"] * cfg3["E"])
            out[name]["stream_k_groups"] = R.router_tc_groups(M, cfg3["H"], cfg3["E"], cfg3["k"])
        except Exception as e:  # a detail row never costs the headline line
            out[name] = {"error": str(e)[:200]}
    return out


def run_only(args):
    """Run one workload's router calls and print its per-call time (for
    profiling the kernel of one configuration under ncu)."""
    import torch

    from moe_expert_router_02_gb300 import synth
    C = synth.CONFIGS
    table = {
        "decode": lambda: RouterSet(C["C1"], 8, LAYERS),
        "decode_m1": lambda: RouterSet(C["C1"], 1, LAYERS),
        "sqrtsoftplus_m64": lambda: RouterSet(C["C2"], 64, LAYERS),
        "m2_table": lambda: RouterSet(C["C4"], 2, LAYERS, table=True),
        "prefill_bf16": lambda: RouterSet(C["C3"], C["C3"]["M"], 1, pool_bytes=0),
        "prefill_nvfp4": lambda: RouterSet(C["C3"], C["C3"]["M"], 1, w_dtype=synth.NVFP4,
                                           pool_bytes=0),
    }
    if args.only in ("table_1e5", "gather_1e3"):
        from moe_expert_router_02_gb300 import router as R
        k = C["C4"]["k"]
        G = C["C4"]["table_groups"] if args.only == "table_1e5" else 1000
        idx = dev(synth.table_pairs(G, k, 256, seed=0))
        tb = (torch.empty((G, 2 * k), dtype=torch.int32, device="cuda"),
              torch.empty((G, 2 * k), dtype=torch.uint8, device="cuda"),
              torch.empty((G, 2, k), dtype=torch.uint8, device="cuda"),
              torch.empty((G,), dtype=torch.int32, device="cuda"))
        if args.only == "table_1e5":
            fn = lambda: R.route_table(idx, G, 2, k, *tb)  # noqa: E731
        else:
            D = C["C4"]["H"]
            R.route_table(idx, G, 2, k, *tb)
            y, w, sh = synth.gather_inputs(G, k, D, seed=0)
            yd, wd, sd = dev(y.view(np.int16)), dev(w), dev(sh.view(np.int16))
            od = torch.empty((G, 2, D), dtype=torch.int16, device="cuda")
            fn = lambda: R.route_gather_add(yd, tb[2], wd, sd, G, 2, k, D, od)  # noqa: E731
        ms = time_graph(fn, args.steps, warm=args.warmup)
        print(json.dumps({"workload": args.only, "us_per_call": ms * 1e3, "steps": args.steps}))
        torch.cuda.synchronize()
        return
    rs = table[args.only]()
    rs.capture()
    ms = time_graph(rs.step, args.steps, warm=args.warmup)
    print(json.dumps({"workload": args.only, "us_per_call": ms * 1e3 / rs.calls,
                      "calls_per_step": rs.calls, "steps": args.steps}))
    torch.cuda.synchronize()


def run_phase_stamps(args):
    """Per-phase latency of the decode kernel from the measurement build's
    %globaltimer stamps (moe_expert_router_02_gb300/build.py, variant
    "stamps"): the 40-call decode graph replayed, then the median over calls
    of each phase (ns). Prints one JSON line."""
    import torch

    from moe_expert_router_02_gb300 import router as R
    from moe_expert_router_02_gb300 import synth
    R.use_variant("stamps")
    M = args.stamps_m
    cfg = dict(synth.CONFIGS[args.stamps_config])
    if args.stamps_sigmoid:
        cfg["act"] = synth.SIGMOID
    rs = RouterSet(cfg, M, LAYERS)
    rs.capture()
    for _ in range(args.warmup):
        rs.step()
    torch.cuda.synchronize()
    R.phase_stamps()  # clears the launch counters
    reps = 6  # 240 calls, inside the 256 stamp slots
    for _ in range(reps):
        rs.step()
    torch.cuda.synchronize()
    st, sel, refines = R.phase_stamps(with_refines=True)
    st, sel = st.astype(np.int64), sel.astype(np.int64)
    n = reps * LAYERS
    # the measurement build stamps the first row group's cluster (4 rows up
    # to M=24, 8 up to M=32, else 16); its CTAs c < rows select a row each
    rows = min(M, 4 if M <= 24 else 8 if M <= 32 else 16)
    own = [c for c in range(16) if c < rows]
    ph = {k: [] for k in ("prev_end_to_wait_return", "wait_return_to_w_ready",
                          "w_ready_to_partials", "partials_to_sent", "sent_to_rows_landed",
                          "rows_landed_to_selected", "wait_return_to_last_selected",
                          "call_period", "start_before_prev_end")}
    for c in range(1, n):
        cur, prev = st[c], st[c - 1]
        prev_end = prev[own, 7].max()
        w2 = cur[:, 2].min()
        ph["prev_end_to_wait_return"].append(w2 - prev_end)
        ph["wait_return_to_w_ready"].append(np.median(cur[:, 3] - cur[:, 2]))
        ph["w_ready_to_partials"].append(np.median(cur[:, 4] - cur[:, 3]))
        ph["partials_to_sent"].append(np.median(cur[:, 5] - cur[:, 4]))
        ph["sent_to_rows_landed"].append(np.median(cur[own, 6] - cur[:, 5].max()))
        ph["rows_landed_to_selected"].append(np.median(cur[own, 7] - cur[own, 6]))
        ph["wait_return_to_last_selected"].append(cur[own, 7].max() - w2)
        ph["call_period"].append(cur[own, 7].max() - prev_end)
        ph["start_before_prev_end"].append(prev_end - cur[:, 0].min())
    res = {k: float(np.median(v)) for k, v in ph.items()}
    # the last call's selection, sub-phase by sub-phase (selecting CTAs)
    sub = np.diff(sel[own], axis=1)
    res_sel = {n_: float(np.median(sub[:, i])) for i, n_ in
               enumerate(("sort", "rounds", "weights", "stores"))}
    res_sel["entry_to_packed"] = float(np.median(sel[own, 0] - st[n - 1][own, 6]))
    act = {synth.SOFTMAX: "softmax", synth.SQRT_SOFTPLUS: "sqrt-softplus + bias",
           synth.SIGMOID: "sigmoid + bias"}[cfg["act"]]
    print(json.dumps({"workload": f"single-cluster router M={M}, H={cfg['H']}, E={cfg['E']}, "
                                  f"k={cfg['k']}, {act}, 40-call graph, first row group "
                                  f"({rows} rows)",
                      "calls": n - 1, "median_ns": res, "selection_ns": res_sel,
                      "rows_selected": n * M, "rows_reranked": refines[0],
                      "rows_fp64": refines[1], "rows_pair_rounds": refines[2]}))


def run_phase_stamps_split(args):
    """Per-phase latency of the split-cluster kernel (measurement build) on
    the sqrt-softplus + bias router at M=64, H=4096, E=256, k=6 (40-call
    graph): medians over calls of each phase (ns). Prints one JSON line."""
    import torch

    from moe_expert_router_02_gb300 import router as R
    from moe_expert_router_02_gb300 import synth
    R.use_variant("stamps")
    rs = RouterSet(synth.CONFIGS["C2"], 64, LAYERS)
    rs.capture()
    for _ in range(args.warmup):
        rs.step()
    torch.cuda.synchronize()
    R.split_phase_stamps()  # clears the launch counters
    R.phase_stamps()  # and the re-rank counts
    rs.step()  # 40 calls, inside the 64 stamp slots
    torch.cuda.synchronize()
    st = R.split_phase_stamps().astype(np.int64)
    names = ("wait_return_to_w_ready", "w_ready_to_partials", "partials_to_slices_ready",
             "slices_to_logits_stored", "logits_to_barrier", "barrier_to_ticket_known")
    ph = {n: [] for n in names + ("prev_end_to_wait_return", "ticket_to_selected",
                                   "wait_return_to_selected", "call_period")}
    prev_end = None
    ph["last_cluster_ticket_after_median"] = []
    for c in range(LAYERS):
        cur = st[c]
        live = cur[:, 0] > 0
        # the last cluster's CTAs: a selection stamp of this call (after its
        # ticket stamp); other slots keep stamps of earlier calls
        sel = live & (cur[:, 9] > cur[:, 8]) & (cur[:, 8] > 0)
        if sel.any():
            ph["last_cluster_ticket_after_median"].append(
                np.median(cur[sel, 7]) - np.median(cur[live, 7]))
        end = cur[sel, 9].max() if sel.any() else None
        w2 = cur[live, 2].min()
        if prev_end is not None and end is not None:
            ph["prev_end_to_wait_return"].append(w2 - prev_end)
            ph["call_period"].append(end - prev_end)
        for i, n_ in enumerate(names):
            ph[n_].append(np.median(cur[live, i + 3] - cur[live, i + 2]))
        if sel.any():
            ph["ticket_to_selected"].append(np.median(cur[sel, 9] - cur[sel, 8]))
            ph["wait_return_to_selected"].append(end - w2)
        prev_end = end
    # the last call's selection, sub-phase by sub-phase: lane 0 of the last
    # warp of each of the selecting cluster's CTAs to select a row
    _, ss, refines = R.phase_stamps(with_refines=True)
    ss = ss.astype(np.int64)
    cl = int(sel.sum())
    last = st[LAYERS - 1]
    sel_rows = np.nonzero((last[:, 9] > last[:, 8]) & (last[:, 8] > 0))[0]
    ranks = [int(c) % cl for c in sel_rows] if cl else []
    res_sel = {}
    if ranks:
        sub = np.diff(ss[ranks], axis=1)
        res_sel = {n_: float(np.median(sub[:, i])) for i, n_ in
                   enumerate(("sort", "rounds", "weights", "stores"))}
        res_sel["entry_to_packed"] = float(np.median(ss[ranks, 0] - last[sel_rows, 8]))
    print(json.dumps({"workload": "split-cluster router M=64, H=4096, E=256, k=6, "
                                  "sqrt-softplus + bias, 40-call graph",
                      "median_ns": {k: float(np.median(v)) for k, v in ph.items() if v},
                      "selection_ns": res_sel, "rows_selected": 64 * LAYERS,
                      "rows_reranked": refines[0], "rows_fp64": refines[1]}))


def run_phase_stamps_prefill(args):
    """Per-CTA phase timeline of the prefill kernel (measurement build) on
    the M=16384, H=7168, E=256, k=8 sqrt-softplus + bias workload: each
    phase's median and largest time from the launch's first CTA start (us),
    and the CTAs that re-ranked near ties. Prints one JSON line."""
    import torch

    from moe_expert_router_02_gb300 import router as R
    from moe_expert_router_02_gb300 import synth
    R.use_variant("stamps")
    cfg = synth.CONFIGS["C3"]
    w_dtype = synth.NVFP4 if args.stamps_nvfp4 else None
    rs = RouterSet(cfg, args.stamps_prefill_m, 1, w_dtype=w_dtype, pool_bytes=0)
    rs.capture()
    out = []
    for rep in range(args.steps):
        rs.step()
        torch.cuda.synchronize()
        st = R.tc_phase_stamps().astype(np.int64)
        live = st[:, 0] > 0
        st = st[live]
        t0 = st[:, 0].min()
        names = ["entry", "setup", "epi_setup", "acc_complete", "partials_added", "pass_a",
                 "pass_bc", "merged", "stored", "cta_end"]
        rel = (st[:, :10] - t0) / 1e3
        ent = {n: {"median": float(np.median(rel[:, i])), "max": float(rel[:, i].max())}
               for i, n in enumerate(names)}
        fm = st[:, 11][st[:, 11] > 0]
        ent["first_mma"] = {"median": float(np.median((fm - t0) / 1e3)),
                            "max": float(((fm - t0) / 1e3).max())}
        fin = st[:, 15] > 0  # CTAs that finished a tile (ran passes A-C)
        for i, n_ in ((12, "threshold"), (13, "pass_b"), (14, "pooled_act"), (15, "inserted")):
            ent[n_] = {"median": float(np.median((st[fin, i] - t0) / 1e3)),
                       "max": float(((st[fin, i] - t0) / 1e3).max())}
        ent["cand_thread0"] = {"median": float(np.median(st[fin, 16])),
                               "max": int(st[fin, 16].max())}
        ent["cand_warp0_total"] = {"median": float(np.median(st[fin, 17])),
                                   "max": int(st[fin, 17].max())}
        ref = np.nonzero(st[:, 10] == 1)[0]
        ent["refined_ctas"] = [{"cta": int(c), "end": float(rel[c, 9])} for c in ref]
        ent["ctas"] = int(live.sum())
        ent["slowest"] = [{"cta": int(c), "end": float(rel[c, 9]),
                           "acc": float(rel[c, 3]), "refined": int(st[c, 10])}
                          for c in np.argsort(-rel[:, 9])[:6]]
        if args.stamps_dump:  # per CTA: SM, plan, accumulator complete, end (us)
            def us(col):
                return [round(float(v - t0) / 1e3, 3) if v > 0 else None for v in st[:, col]]
            ent["per_cta"] = {"sm": st[:, 18].tolist(), "plan": st[:, 19].tolist(),
                              "acc": [round(float(v), 3) for v in rel[:, 3]],
                              "parts": [round(float(v), 3) for v in rel[:, 4]],
                              "end": [round(float(v), 3) for v in rel[:, 9]],
                              "accp": us(20), "published": us(21), "prefetched": us(22),
                              "last_mma": us(23), "b0_flag": us(24), "b0_landed": us(25),
                              "b0_added": us(26), "bl_flag": us(27), "bl_landed": us(28),
                              "bl_added": us(29),
                              "refine": [[us(30 + 4 * q)[c], us(31 + 4 * q)[c], us(32 + 4 * q)[c],
                                          int(st[c, 33 + 4 * q])] for c in range(len(st))
                                         for q in range(4) if st[c, 30 + 4 * q] > 0]}
        out.append(ent)
    print(json.dumps({"workload": f"prefill M={args.stamps_prefill_m}, H=7168, E=256, k=8, "
                                  f"sqrt-softplus + bias, {'NVFP4' if w_dtype else 'BF16'} W",
                      "launches": out}))


def run_reference(args, rank, world):
    """CPU oracle on the headline workload (rank 0 only)."""
    if rank != 0:
        return
    from moe_expert_router_02_gb300 import synth
    import oracle
    cfg = synth.CONFIGS["C1"]
    M = 8
    case = synth.make_case(cfg, M=M, seed=0)
    for _ in range(args.warmup):
        oracle.router(case)
    t0 = time.perf_counter()
    per_step = max(1, args.ref_calls)
    for _ in range(args.steps):
        for _ in range(per_step):
            oracle.router(case)
    dt = time.perf_counter() - t0
    value = M * per_step * args.steps / dt
    line = {
        "impl": "reference",
        "metric": "router tokens/s (decode M=8, H=2048, E=256, top-8 softmax, 40 layers)",
        "value": value, "unit": "router tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": dt * 1e3 / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "decode router: M=8 rows, H=2048, E=256, k=8, softmax; "
                               f"each step = {per_step} oracle router calls (sample of the 40 "
                               "layer calls)"},
        "cpu_baseline": {"value": value, "unit": "router tokens/s", "cores": 1, "kind": "oracle",
                         "sample": f"{per_step} calls per step x {args.steps} steps, single thread"},
        "e2e": {"value": value, "unit": "router tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--quick", action="store_true", help="headline only, no per-config detail")
    ap.add_argument("--cpu-budget", type=float, default=10.0)
    ap.add_argument("--ref-calls", type=int, default=8)
    ap.add_argument("--phase-stamps", action="store_true",
                    help="per-phase latency of the decode kernel (measurement build)")
    ap.add_argument("--stamps-m", type=int, default=8)
    ap.add_argument("--stamps-config", default="C1", choices=["C1", "C2"],
                    help="--phase-stamps: decode softmax (C1) or sqrt-softplus + bias (C2)")
    ap.add_argument("--stamps-sigmoid", action="store_true",
                    help="--phase-stamps: the sigmoid + bias score on the chosen config")
    ap.add_argument("--phase-stamps-split", action="store_true",
                    help="per-phase latency of the split-cluster kernel (measurement build)")
    ap.add_argument("--phase-stamps-prefill", action="store_true",
                    help="per-CTA phase timeline of the prefill kernel (measurement build)")
    ap.add_argument("--stamps-prefill-m", type=int, default=16384)
    ap.add_argument("--stamps-nvfp4", action="store_true")
    ap.add_argument("--stamps-dump", action="store_true",
                    help="--phase-stamps-prefill: add per-CTA SM, plan and times")
    ap.add_argument("--only", default=None,
                    choices=["decode", "decode_m1", "sqrtsoftplus_m64", "m2_table",
                             "prefill_bf16", "prefill_nvfp4", "table_1e5", "gather_1e3"],
                    help="run one workload's calls only (profiling)")
    args = ap.parse_args()
    if args.only:
        run_only(args)
        return
    if args.phase_stamps:
        run_phase_stamps(args)
        return
    if args.phase_stamps_prefill:
        run_phase_stamps_prefill(args)
        return
    if args.phase_stamps_split:
        run_phase_stamps_split(args)
        return
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    rank, world, local = dist_setup(args.gpus)
    run_ours(args, rank, world, local)


if __name__ == "__main__":
    main()
