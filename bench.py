"""Benchmark of the NVFP4 MoE layer on GB300 (one JSON line on stdout).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config decode] [--impl ours|reference]

A step is one pass of the whole layer (route, permute, quantize, gate_up GEMM
with fused SiLU*up requant, down GEMM, combine; BF16 output) over one batch.
Default workload: the 30B-A3B-shaped decode layer (T=32, H=2048, I=768, E=128,
top-8), whose weight-streaming gate_up GEMM carries the headline roofline
(fraction of HBM).  The same line carries a `prefill` object: the 4096-token
prefill of the same layer (same weights), timed in the same process, with the
grouped GEMMs' fraction of the dense FP4 tensor peak.  Inputs are synthetic
(seeded: activations and logits from the CPU generator, weights drawn on the
device and prepared by the library before timing).  The timed region replays a
CUDA graph of the K steps; the weights streamed per step (about 300 MB) exceed
the 129 MB L2.

Multi-GPU: every rank runs its own replica on its own batch (the layer shards
by tokens with no exchange): value = tokens of all ranks / max-over-ranks time.

--impl reference times the CPU oracle (the reference arm for this build) on a
bounded token sample of the same workload, on the host cores.
"""
import os

os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")   # the oracle baseline runs on one core
os.environ.setdefault("OMP_NUM_THREADS", "1")
os.environ.setdefault("MKL_NUM_THREADS", "1")

import argparse  # noqa: E402
import json  # noqa: E402
import statistics  # noqa: E402
import subprocess  # noqa: E402
import sys  # noqa: E402
import tempfile  # noqa: E402
import time  # noqa: E402

import numpy as np  # noqa: E402
import torch  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from synth import CONFIGS, expert_weights, make_inputs  # noqa: E402

METRIC = "NVFP4 MoE layer tokens/s; grouped-GEMM % FP4 TC peak (prefill) / % HBM (decode)"
# (name, first event, last event) of the forward's six stage events; events 1 and 2
# bracket the separate activation quantization, which the route kernel now does.
STAGES = [("route_permute_quant_a1", 0, 1), ("gate_up_gemm_swiglu_quant", 2, 3), ("down_gemm", 3, 4),
          ("combine", 4, 5)]


def kernels_per_step(T):
    """Kernels one forward launches: top-k, (prefix for > 256 tokens), permute+quantize,
    gate_up GEMM, down GEMM, combine."""
    return 1 + (1 if (T + 31) // 32 > 8 else 0) + 1 + 2 + 1


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d.get("hbm_gbs", 6800.0), d.get("bf16_tflops", 1900.0), "measured"
    return 6800.0, 1900.0, "fallback"


def activation_scales(name):
    d = json.load(open(os.path.join(ROOT, "tests", "golden", "activation_scales.json")))
    return d[name]["gs_a1"], d[name]["gs_a2"]


def layer_bytes(cfg, counts):
    """Algorithmic bytes of one step (intermediates excluded): codes and block
    scales of the touched experts' w13 and w2, their two FP32 global scales,
    x (bf16), logits (fp32) and out (bf16).  counts: rows per expert (shared
    included)."""
    touched = int((np.asarray(counts) > 0).sum())
    per_expert = 3 * cfg.H * cfg.I * (0.5 + 1.0 / 16) + 8
    return touched, touched * per_expert + cfg.T * cfg.H * 2 + cfg.T * cfg.E * 4 + cfg.T * cfg.H * 2


def gemm1_bytes(cfg, touched):
    """Algorithmic bytes of the gate_up GEMM launch: codes, block scales and
    global scale of the touched experts' w13 (the A1 / A2 intermediates are an
    implementation cost, not counted)."""
    return touched * (2 * cfg.I * cfg.H * (0.5 + 1.0 / 16) + 4)


def gemm2_bytes(cfg, touched):
    """Algorithmic bytes of the down GEMM launch: the touched experts' w2."""
    return touched * (cfg.H * cfg.I * (0.5 + 1.0 / 16) + 4)


class ClockSampler:
    def __init__(self, path):
        self.path = path
        self.proc = None

    def start(self):
        q = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        dev = os.environ.get("LOCAL_RANK", "0")
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", dev, f"--query-gpu={q}", "--format=csv,noheader,nounits",
                                          "-lms", "50"], stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        self.proc.terminate()
        self.proc.wait()
        self.f.close()
        rows = [r.split(", ") for r in open(self.path).read().strip().splitlines() if r.count(",") >= 8]
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                s, m, pw = float(r[1]), float(r[2]), float(r[3])
            except ValueError:
                continue
            mx = m
            if pw > 200:           # under load
                sm.append(s)
                for n, v in zip(names, r[5:9]):
                    if v.strip().lower() == "active":
                        reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples_under_load": len(sm)}


def oracle_sample(cfg, x, logits, bias, tokens, oracle_w):
    from oracle import moe as M
    xs = x[tokens].float().cpu().numpy()
    ls = logits[tokens].cpu().numpy()
    b = None if bias is None else bias.cpu().numpy()
    E = cfg.E_total
    gs1, gs2 = activation_scales(cfg.name)
    return M.moe_forward(xs, ls, b, cfg.k, cfg.renormalize, cfg.shared, lambda e: oracle_w[e],
                         np.full(E, gs1, np.float32), np.full(E, gs2, np.float32))


# ----------------------------------------------------------------------------- CPU oracle baseline
# Each worker process holds its own copy of the layer's inputs and of the oracle's
# quantized weights for the experts its token visits (drawn from the CPU
# generator: the same recipe; the oracle's time does not depend on the values).
_ORACLE = {}


def _oracle_state(cfg_name, seed, token):
    from oracle import moe as M
    key = (cfg_name, seed)
    if key not in _ORACLE:
        cfg = CONFIGS[cfg_name]
        x, logits, bias = make_inputs(cfg, seed, device="cpu")
        _ORACLE[key] = (cfg, x, logits, bias, {})
    cfg, x, logits, bias, ow = _ORACLE[key]
    ids, _ = M.route(logits[[token]].numpy(), None if bias is None else bias.numpy(), cfg.k, cfg.renormalize)
    for e in sorted(set(ids.reshape(-1).tolist()) | ({cfg.E} if cfg.shared else set())):
        if e not in ow:
            w13, w2 = expert_weights(cfg, e, seed, device="cpu")
            ow[e] = (*M.quantize_expert_weights(w13.numpy()), *M.quantize_expert_weights(w2.numpy()))
    return _ORACLE[key]


def _oracle_job(args):
    """One worker's share: (passes, seconds) of oracle forwards over one token
    (steps S1-S7; weights prepared before the clock starts).  budget_s > 0: as
    many passes as fit; budget_s == 0: set-up only; budget_s < 0: one pass."""
    cfg_name, seed, token, budget_s = args
    cfg, x, logits, bias, ow = _oracle_state(cfg_name, seed, token)
    if budget_s == 0:
        return 0, 0.0
    t0 = time.perf_counter()
    n = 0
    while True:
        oracle_sample(cfg, x, logits, bias, [token], ow)
        n += 1
        dt = time.perf_counter() - t0
        if budget_s < 0 or dt >= budget_s:
            return n, dt


def cpu_model():
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    for line in open("/proc/cpuinfo"):
        if line.startswith("model name"):
            return line.split(":", 1)[1].strip()
    import platform
    return platform.machine()


def oracle_pool(cores):
    import multiprocessing as mp
    return mp.get_context("spawn").Pool(cores)


def cpu_oracle_rates(cfg, seed, budget_s):
    """Oracle tokens/s on one core (token 0) and on every core (one token per
    core, tokens 0 .. cores-1), each worker single-threaded."""
    cores = os.cpu_count() or 1
    with oracle_pool(cores) as pool:
        pool.map(_oracle_job, [(cfg.name, seed, t % cfg.T, 0) for t in range(cores)], chunksize=1)
        n1, dt1 = pool.apply(_oracle_job, ((cfg.name, seed, 0, budget_s),))
        res = pool.map(_oracle_job, [(cfg.name, seed, t % cfg.T, budget_s) for t in range(cores)], chunksize=1)
    one = n1 / dt1
    allc = sum(n / dt for n, dt in res)
    sample = (f"oracle forwards (S1-S7) over single tokens of the {cfg.name} batch, weights prepared "
              f"beforehand: token 0 on one core for {dt1:.1f} s ({n1} passes); tokens 0-{cores - 1}, "
              f"one per core, for {budget_s:.0f} s ({sum(n for n, _ in res)} passes)")
    return {"value": allc, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": sample,
            "one_core": one, "cpu_model": cpu_model()}


def job_time_and_value(elapsed_ms, T, K, dist, device):
    """Whole-job timing of K steps of T tokens on every rank: the slowest rank's
    time (max over ranks) and the tokens all ranks processed per second."""
    t = torch.tensor([float(elapsed_ms)], device=device)
    world = 1
    if dist is not None:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        world = dist.get_world_size()
    ms = float(t.item())
    return ms, T * K * world / (ms * 1e-3)


def workload_config(cfg, world):
    """The `config` object both arms report for workload `cfg`."""
    return {"workload": f"{cfg.name}: {cfg.description} (T={cfg.T} H={cfg.H} I={cfg.I} E={cfg.E}"
                        f"{'+1 shared' if cfg.shared else ''} top-{cfg.k})",
            "T": cfg.T, "H": cfg.H, "I": cfg.I, "E": cfg.E, "k": cfg.k, "shared": cfg.shared,
            "parallelism": f"replicas x{world}", "l2": "inputs larger than L2 (weights streamed per step)"}


def run_reference(args, cfg):
    """The reference arm: the CPU oracle as it stands, on every host core (one
    token per core and step, each worker single-threaded; weights prepared
    before timing).  A step is one oracle forward over `cores` tokens of the
    workload; value = tokens / mean step time."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    seed = 0
    cores = os.cpu_count() or 1
    jobs = [(cfg.name, seed, t % cfg.T, -1.0) for t in range(cores)]
    with oracle_pool(cores) as pool:
        pool.map(_oracle_job, [(n, s_, t, 0) for n, s_, t, _ in jobs], chunksize=1)   # set-up, untimed
        for _ in range(args.warmup):
            pool.map(_oracle_job, jobs, chunksize=1)
        times = []
        for _ in range(args.steps):
            t0 = time.perf_counter()
            pool.map(_oracle_job, jobs, chunksize=1)
            times.append(time.perf_counter() - t0)
    ms = 1000 * statistics.mean(times)
    value = cores / (ms / 1000)
    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": dict(workload_config(cfg, args.gpus), sample_tokens=cores,
                           timing="oracle on the host cores, wall clock; a step is one forward of "
                                  f"{cores} tokens, one per core"),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": f"tokens 0-{cores - 1} of the {cfg.name} batch through the CPU oracle "
                                       "(S1-S7), one token per core per step", "cpu_model": cpu_model()},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


DENSE_N, DENSE_K = 34816, 5120
DENSE_M = (1, 16, 64, 256, 1024, 4096)


def dense_sweep(args):
    """The dense NVFP4 W4A4 linear of the pages' second workload: gate_up with
    N = 34816, K = 5120 for M = 1..4096 tokens.  One call = quantize the BF16
    activations (TILED_GROUPED, one group) + the grouped GEMM with one group,
    FP32 out.  The K calls are one CUDA graph; three weight copies (3 x 100 MB,
    more than L2) rotate so that the weights stream from HBM.  One JSON line
    per M, with the fraction of the measured HBM copy rate (weights) and of the
    dense FP4 tensor peak (measured bf16 x 6)."""
    import nvfp4_moe_grouped_router_gb300 as nvf
    from nvfp4_moe_grouped_router_gb300 import build as nvf_build
    torch.cuda.set_device(0)
    nvf_build.build()
    nvf.lib()
    hbm, bf16, src = load_peaks()
    N, K = DENSE_N, DENSE_K
    g = torch.Generator(device="cuda").manual_seed(0)
    copies = []
    for _ in range(3):
        w = torch.randn(N, K, generator=g, device="cuda") * 0.02
        gs_w = torch.tensor([w.abs().max().item() / 2688.0], dtype=torch.float32, device="cuda")
        B, _ = nvf.quantize(w, gs_w, layout=nvf.LAYOUT_TILED)
        copies.append((B, gs_w))
        del w
    w_bytes = nvf.tiled_bytes(N, 0, K)
    stream = torch.cuda.Stream()
    for Mr in DENSE_M:
        a = torch.randn(Mr, K, generator=g, device="cuda").to(torch.bfloat16)
        gs_a = torch.tensor([a.float().abs().max().item() / 2688.0], dtype=torch.float32, device="cuda")
        offs = torch.tensor([0, Mr], dtype=torch.int32, device="cuda")
        tiles = torch.tensor([0, (Mr + 127) // 128], dtype=torch.int32, device="cuda")
        A = torch.zeros(nvf.tiled_bytes(Mr, 1, K), dtype=torch.uint8, device="cuda")
        D = torch.empty(Mr, N, dtype=torch.float32, device="cuda")

        def call(i):
            B, gs_w = copies[i % 3]
            nvf.quantize(a, gs_a, layout=nvf.LAYOUT_TILED_GROUPED, offsets=offs, tile_offsets=tiles, codes=A)
            nvf.grouped_gemm(A, Mr, B, gs_a, gs_w, offs, tiles, N, K, D=D)

        steps = max(3, min(args.steps, 60 if Mr >= 1024 else 300))
        for i in range(max(3, args.warmup)):
            call(i)
        torch.cuda.synchronize()
        stream.wait_stream(torch.cuda.current_stream())
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for i in range(steps):
                call(i)
        torch.cuda.current_stream().wait_stream(stream)
        graph.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        graph.replay()
        e1.record()
        torch.cuda.synchronize()
        code, detail = nvf.device_status()
        if code != 0:
            raise RuntimeError(f"device error word {code} at {detail}")
        us = e0.elapsed_time(e1) * 1e3 / steps
        tflops = 2.0 * Mr * N * K / (us * 1e-6) / 1e12
        gbs = (w_bytes + Mr * K * 2 + Mr * N * 4) / (us * 1e-6) / 1e9
        print(json.dumps({"metric": "dense NVFP4 W4A4 linear (gate_up N=34816 K=5120): us per call", "M": Mr,
                          "us_per_call": us, "tflops": tflops, "gbs": gbs, "hbm_frac": gbs / hbm,
                          "tc_frac_fp4": tflops / (6.0 * bf16), "peak_source": src, "steps": steps,
                          "launches_per_call": 2, "data": "synthetic", "l2": "3 weight copies rotate (300 MB)"}),
              flush=True)


def router_sweep(args):
    """The router gate (the step before routing) on the bench layer's shape:
    x bf16 [T, 2048] . w_gate bf16 [129, 2048]^T (128 routed experts + one
    shared-expert gate row) for the decode and prefill batches.  One JSON line
    per T with the time per call (CUDA graph of the calls), the bf16 FLOP rate
    and the bytes moved (x, w_gate, logits) against the measured peaks."""
    import nvfp4_moe_grouped_router_gb300 as nvf
    from nvfp4_moe_grouped_router_gb300 import build as nvf_build
    torch.cuda.set_device(0)
    nvf_build.build()
    nvf.lib()
    hbm, bf16, src = load_peaks()
    H, n = 2048, 129
    g = torch.Generator().manual_seed(0)
    w = (torch.randn(n, H, generator=g) * 0.02).to(torch.bfloat16).cuda()
    stream = torch.cuda.Stream()
    for T in (32, 4096):
        x = torch.randn(T, H, generator=g).to(torch.bfloat16).cuda()
        lg = torch.empty(T, n, device="cuda")
        steps = max(3, min(args.steps, 500))
        for _ in range(max(3, args.warmup)):
            nvf.router_gemm(x, w, logits=lg)
        torch.cuda.synchronize()
        stream.wait_stream(torch.cuda.current_stream())
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for _ in range(steps):
                nvf.router_gemm(x, w, logits=lg)
        torch.cuda.current_stream().wait_stream(stream)
        graph.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        graph.replay()
        e1.record()
        torch.cuda.synchronize()
        code, detail = nvf.device_status()
        if code != 0:
            raise RuntimeError(f"device error word {code} at {detail}")
        us = e0.elapsed_time(e1) * 1e3 / steps
        nbytes = T * H * 2 + n * H * 2 + T * n * 4
        print(json.dumps({"metric": "router gate x . w_gate^T (bf16, H=2048, 128 + 1 rows): us per call", "T": T,
                          "us_per_call": us, "tflops": 2.0 * T * H * n / (us * 1e-6) / 1e12,
                          "tc_frac_bf16": 2.0 * T * H * n / (us * 1e-6) / 1e12 / bf16,
                          "gbs": nbytes / (us * 1e-6) / 1e9, "hbm_frac": nbytes / (us * 1e-6) / 1e9 / hbm,
                          "peak_source": src, "steps": steps, "launches_per_call": 1, "data": "synthetic"}),
              flush=True)


def _graph_time_us(fn, steps, warmup):
    """Mean microseconds per call of fn, replayed as one CUDA graph of `steps` calls."""
    for _ in range(max(3, warmup)):
        fn(0)
    torch.cuda.synchronize()
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for i in range(steps):
            fn(i)
    torch.cuda.current_stream().wait_stream(stream)
    graph.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    graph.replay()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) * 1e3 / steps


def w4a16_sweep(args):
    """The weight-only path (FP16 or BF16 activations x NVFP4 weights
    dequantized in the kernel) beside the W4A4 GEMM on the same weight bytes: (1) the decode layer's
    gate_up GEMM (its routing's expert groups, x gathered in permuted order and
    rounded to FP16); (2) the pages' dense gate_up shape N = 34816, K = 5120,
    three weight copies rotating so that weights stream from HBM.  One JSON line
    per case."""
    import nvfp4_moe_grouped_router_gb300 as nvf
    from nvfp4_moe_grouped_router_gb300 import build as nvf_build
    torch.cuda.set_device(0)
    nvf_build.build()
    nvf.lib()
    hbm, bf16, src = load_peaks()
    steps = max(3, min(args.steps, 200))
    cfg = CONFIGS["decode"]
    w = nvf.prepare_weights(cfg.E, cfg.H, cfg.I, cfg.shared, lambda e: expert_weights(cfg, e, 0, device="cuda"))
    x, logits, _ = make_inputs(cfg, 0, device="cpu")
    x, logits = x.cuda(), logits.cuda()
    r = nvf.route_permute(logits, cfg.k)
    offs, tiles = r["expert_offsets"], r["tile_offsets"]
    touched = int((offs[1:] > offs[:-1]).sum().item())
    A = x[r["perm_token"].long()].to(torch.float16).contiguous()
    D = torch.empty(cfg.R, 2 * cfg.I, device="cuda")
    us = _graph_time_us(lambda i: nvf.w4a16_grouped_gemm(A, w.w13, w.gs_w13, offs, tiles, 2 * cfg.I, cfg.H, D=D),
                        steps, args.warmup)
    nbytes = gemm1_bytes(cfg, touched)
    print(json.dumps({"metric": "W4A16 grouped GEMM, decode layer gate_up (N=1536, K=2048, 256 rows in "
                                f"{touched} experts): us per call", "us_per_call": us,
                      "gbs": nbytes / (us * 1e-6) / 1e9, "hbm_frac": nbytes / (us * 1e-6) / 1e9 / hbm,
                      "algorithmic_bytes": nbytes, "peak_source": src, "steps": steps}), flush=True)
    # the same call on the BF16 rows as they come (the kernel rounds them to FP16)
    A_bf = x[r["perm_token"].long()].to(torch.bfloat16).contiguous()
    us = _graph_time_us(lambda i: nvf.w4a16_grouped_gemm(A_bf, w.w13, w.gs_w13, offs, tiles, 2 * cfg.I, cfg.H, D=D),
                        steps, args.warmup)
    print(json.dumps({"metric": "W4A16 grouped GEMM, decode layer gate_up, BF16 activations: us per call",
                      "us_per_call": us, "gbs": nbytes / (us * 1e-6) / 1e9,
                      "hbm_frac": nbytes / (us * 1e-6) / 1e9 / hbm, "algorithmic_bytes": nbytes,
                      "peak_source": src, "steps": steps}), flush=True)
    del w
    N, K = DENSE_N, DENSE_K
    g = torch.Generator(device="cuda").manual_seed(0)
    copies = []
    for _ in range(3):
        wd = torch.randn(N, K, generator=g, device="cuda") * 0.02
        gs_w = torch.tensor([wd.abs().max().item() / 2688.0], dtype=torch.float32, device="cuda")
        B, _ = nvf.quantize(wd, gs_w, layout=nvf.LAYOUT_TILED)
        copies.append((B, gs_w))
        del wd
    w_bytes = nvf.tiled_bytes(N, 0, K)
    for Mr in DENSE_M:
        a = torch.randn(Mr, K, generator=g, device="cuda").to(torch.bfloat16).to(torch.float16)
        o = torch.tensor([0, Mr], dtype=torch.int32, device="cuda")
        t = torch.tensor([0, (Mr + 127) // 128], dtype=torch.int32, device="cuda")
        Dd = torch.empty(Mr, N, device="cuda")
        n = steps if Mr < 1024 else min(steps, 40)
        us = _graph_time_us(lambda i: nvf.w4a16_grouped_gemm(a, copies[i % 3][0], copies[i % 3][1], o, t, N, K, D=Dd),
                            n, args.warmup)
        tflops = 2.0 * Mr * N * K / (us * 1e-6) / 1e12
        gbs = (w_bytes + Mr * K * 2 + Mr * N * 4) / (us * 1e-6) / 1e9
        print(json.dumps({"metric": "W4A16 dense linear (gate_up N=34816 K=5120): us per call", "M": Mr,
                          "us_per_call": us, "tflops": tflops, "tc_frac_bf16": tflops / bf16, "gbs": gbs,
                          "hbm_frac": gbs / hbm, "peak_source": src, "steps": n}), flush=True)


def ep_sweep(args):
    """Expert parallelism over G ranks, emulated on one GPU: every rank holds
    the workload's batch (seeded per rank), routes it over all experts and
    dispatches; rank 0 receives its segment of every rank's rows, runs its
    E/G experts, returns the rows and combines what comes back.  The exchanges
    are tensor slices here; their bytes are reported.  One JSON line per
    workload: rank 0's device time per step (each a CUDA graph of calls) next
    to the single-device forward of the same batch (all experts local)."""
    import nvfp4_moe_grouped_router_gb300 as nvf
    from nvfp4_moe_grouped_router_gb300 import build as nvf_build
    torch.cuda.set_device(0)
    nvf_build.build()
    nvf.lib()
    G = args.ep
    steps = max(3, min(args.steps, 200))
    for name in ("decode", "prefill"):
        cfg = CONFIGS[name]
        El, H = cfg.E // G, cfg.H
        gs1, gs2 = activation_scales(cfg.name)
        gs_a1 = torch.full((cfg.E_total,), gs1, device="cuda")
        gs_a2 = torch.full((cfg.E_total,), gs2, device="cuda")
        xs, routes, sends = [], [], []
        for r in range(G):
            x, lg, _ = make_inputs(cfg, 1000 + r, device="cpu")
            x, lg = x.cuda(), lg.cuda()
            route = nvf.route_permute(lg, cfg.k, renormalize=cfg.renormalize, shared=cfg.shared)
            xs.append(x)
            routes.append(route)
            sends.append(nvf.ep_dispatch(x, route, cfg.E, cfg.k, cfg.shared, G, r, gs_a1))
        bounds = [np.concatenate([[0], np.cumsum(c.sum(dim=1).cpu().numpy())]) for _, c, _ in sends]
        recv = torch.cat([sends[s][0][bounds[s][0]:bounds[s][1]] for s in range(G)])
        rc = torch.stack([sends[s][1][0] for s in range(G)]).contiguous()
        n = int(rc.sum().item())
        tail = [cfg.E] if cfg.shared else []
        ids = list(range(El)) + tail
        w0 = nvf.prepare_weights(El, H, cfg.I, cfg.shared, lambda j: expert_weights(cfg, ids[j], 0, device="cuda"))
        g = nvf.ep_receive(recv, rc, El, cfg.shared, H, n)
        l1 = nvf.ep_local_scales(gs_a1, cfg.E, G, 0, cfg.shared)
        l2 = nvf.ep_local_scales(gs_a2, cfg.E, G, 0, cfg.shared)
        y = nvf.moe_experts(w0, g["a1"], n, g["offsets"], g["tile_offsets"], l1, l2, torch.bfloat16)
        R = sends[0][2].numel()
        y_back = torch.zeros(R, H, dtype=torch.bfloat16, device="cuda")
        t = {
            "dispatch": _graph_time_us(lambda i: nvf.ep_dispatch(xs[0], routes[0], cfg.E, cfg.k, cfg.shared, G, 0,
                                                                 gs_a1), steps, args.warmup),
            "receive": _graph_time_us(lambda i: nvf.ep_receive(recv, rc, El, cfg.shared, H, n), steps, args.warmup),
            # the down GEMM stores y in received order (row map): no separate return kernel
            "experts": _graph_time_us(lambda i: nvf.moe_experts(w0, g["a1"], n, g["offsets"], g["tile_offsets"], l1,
                                                                l2, torch.bfloat16, y_rows=g["grp_to_recv"]),
                                      steps, args.warmup),
            "combine": _graph_time_us(lambda i: nvf.moe_combine(y_back, routes[0]["topk_w"], sends[0][2], cfg.T,
                                                                cfg.k, cfg.shared), steps, args.warmup),
        }
        del w0
        wf = nvf.prepare_weights(cfg.E, H, cfg.I, cfg.shared, lambda e: expert_weights(cfg, e, 0, device="cuda"))
        lg0 = make_inputs(cfg, 1000, device="cpu")[1].cuda()
        ws = nvf.workspace(cfg.T, wf, cfg.k)
        out = torch.empty(cfg.T, H, dtype=torch.bfloat16, device="cuda")
        single = _graph_time_us(lambda i: nvf.moe_forward(wf, xs[0], lg0, cfg.k, gs_a1, gs_a2,
                                                          renormalize=cfg.renormalize, out=out, ws=ws),
                                steps, args.warmup)
        del wf
        code, detail = nvf.device_status()
        if code != 0:
            raise RuntimeError(f"device error word {code} at {detail}")
        row_bytes = nvf.ep_row_bytes(H)
        print(json.dumps({"metric": f"expert parallelism over {G} ranks, emulated on one GPU: rank 0 device us per step",
                          "workload": name, "G": G, "tokens_per_rank": cfg.T, "rows_sent": R, "rows_received": n,
                          "us": {k: round(v, 2) for k, v in t.items()}, "us_total": round(sum(t.values()), 2),
                          "separate_return_kernel_us": round(_graph_time_us(
                              lambda i: nvf.ep_return(y, g["recv_to_grp"]), steps, args.warmup), 2),
                          "single_device_forward_us": round(single, 2),
                          "exchange_bytes_per_rank": {"dispatch": int(R * row_bytes), "return": int(R * H * 2)},
                          "exchange": "not timed (one GPU)", "steps": steps, "data": "synthetic"}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--config", default="decode", choices=list(CONFIGS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile", action="store_true",
                    help="plain launches of W + K steps and nothing else (for ncu launch lists / captures)")
    ap.add_argument("--dense", action="store_true",
                    help="the dense W4A4 linear sweep (N=34816, K=5120, M=1..4096) instead of the MoE layer")
    ap.add_argument("--router", action="store_true", help="the router gate GEMM at the decode and prefill batches")
    ap.add_argument("--w4a16", action="store_true", help="the weight-only (W4A16) GEMM beside W4A4")
    ap.add_argument("--ep", type=int, default=0, help="expert parallelism over this many ranks, emulated on one GPU")
    args = ap.parse_args()
    if args.ep:
        return ep_sweep(args)
    if args.w4a16:
        return w4a16_sweep(args)
    if args.dense:
        return dense_sweep(args)
    if args.router:
        return router_sweep(args)
    cfg = CONFIGS[args.config]
    if args.impl == "reference":
        return run_reference(args, cfg)

    import nvfp4_moe_grouped_router_gb300 as nvf
    from nvfp4_moe_grouped_router_gb300 import build as nvf_build
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    if rank == 0 or local == 0:
        nvf_build.build()
    if dist:
        dist.barrier()
    nvf.lib()

    seed = 0
    w = nvf.prepare_weights(cfg.E, cfg.H, cfg.I, cfg.shared, lambda e: expert_weights(cfg, e, seed, device="cuda"))
    if args.profile:
        run = LayerRun(nvf, cfg, w, seed + rank)
        for _ in range(max(3, args.warmup) + args.steps):
            run.step()
        run.check()
        print(json.dumps({"profile_run": cfg.name, "steps": args.steps, "warmup": max(3, args.warmup),
                          "kernels_per_step": kernels_per_step(cfg.T)}))
        return

    hbm, bf16, src = load_peaks()
    fp4_peak = bf16 * 6.0           # dense FP4 / BF16 nominal ratio (13.5 / 2.25), TFLOP/s
    K = args.steps
    run = LayerRun(nvf, cfg, w, seed + rank)
    t = run.time(K, args.warmup, dist, rank, e2e=True)
    elapsed_ms, value = job_time_and_value(t["elapsed_ms"], cfg.T, K, dist, "cuda")
    _, e2e_value = job_time_and_value(t["e2e_ms"], cfg.T, t["e2e_steps"], dist, "cuda")
    _, e2e_calls_value = job_time_and_value(t["e2e_eager_ms"], cfg.T, t["e2e_steps"], dist, "cuda")
    touched, lbytes = layer_bytes(cfg, t["counts"])
    ms_step = elapsed_ms / K
    gemms = gemm_rooflines(cfg, t, touched, hbm, fp4_peak, src)
    g1 = gemms["gate_up"]
    roof = {"kernel": "grouped_gemm_kernel<SWIGLU_QUANT> (gate_up GEMM + SiLU*up + NVFP4 requant)",
            "bound": "hbm", "achieved": g1["gbs"], "peak": hbm, "unit": "GB/s", "frac": g1["hbm_frac"],
            "traffic": traffic_from_profiles(cfg.name), "algorithmic_bytes": g1["algorithmic_bytes"],
            "duration_us": g1["us"], "peak_source": f"{src} HBM copy rate (burst)"}
    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "nvfp4 (e2m1 x e2m1, ue4m3 scales, fp32 accumulate) -> bf16",
            "data": "synthetic",
            "config": dict(workload_config(cfg, world),
                           timing="CUDA graph of the K steps (programmatic dependent launch between kernels), "
                                  "CUDA events; stage_ms from a second graph with events at stage boundaries"),
            "stage_ms": t["stage_ms"], "stage_graph_ms_per_step": t["stage_step_ms"],
            "layer_gbs": lbytes / (ms_step * 1e-3) / 1e9,
            "layer_hbm_frac": lbytes / (ms_step * 1e-3) / 1e9 / hbm, "touched_experts": touched,
            "gemms": gemms, "roofline": roof, "clocks": t["clocks"], "gpu_launches": kernels_per_step(cfg.T) * K,
            "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": t["h2d"],
                    "d2h_bytes_per_step": t["d2h"],
                    "path": "nvf_moe_graph_launch: copies in, the layer, copy out as one CUDA graph a step",
                    "separate_calls_value": e2e_calls_value}}
    del run
    if cfg.name == "decode" and world == 1:
        line["prefill"] = prefill_object(nvf, w, seed + rank, min(K, 100), args.warmup, hbm, fp4_peak, src)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_oracle_rates(cfg, seed, budget_s=10.0)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


class LayerRun:
    """Device state of one workload: inputs (activations and logits from the CPU
    generator, uploaded), activation scales, workspace and BF16 output."""

    def __init__(self, nvf, cfg, w, seed):
        self.nvf, self.cfg, self.w = nvf, cfg, w
        x, logits, bias = make_inputs(cfg, seed, device="cpu")
        self.x, self.logits = x.cuda(), logits.cuda()
        self.bias = None if bias is None else bias.cuda()
        gs1, gs2 = activation_scales(cfg.name)
        self.gs_a1 = torch.full((cfg.E_total,), gs1, device="cuda")
        self.gs_a2 = torch.full((cfg.E_total,), gs2, device="cuda")
        self.ws = nvf.workspace(cfg.T, w, cfg.k)
        self.out = torch.empty(cfg.T, cfg.H, dtype=torch.bfloat16, device="cuda")
        self.cw = w.c_struct()

    def step(self, events=None, x=None, logits=None):
        c = self.cfg
        self.nvf.moe_forward(self.w, self.x if x is None else x, self.logits if logits is None else logits, c.k,
                             self.gs_a1, self.gs_a2, bias=self.bias, renormalize=c.renormalize, out=self.out,
                             ws=self.ws, stage_events=events, cw=self.cw)

    def check(self):
        code, detail = self.nvf.device_status()
        if code != 0:
            raise RuntimeError(f"device error word {code} at {detail}")

    def counts(self):
        c = self.cfg
        L = self.nvf.workspace_layout(c.T, c.E, c.H, c.I, c.k, c.shared)
        o = L["expert_offsets"]
        return np.diff(self.ws[o:o + 4 * (c.E_total + 1)].view(torch.int32).cpu().numpy())

    def time(self, K, warmup, dist, rank, e2e=False):
        """K steps replayed as CUDA graphs (kernels chained by programmatic
        dependent launch), timed with CUDA events after a 1 s untimed soak,
        clocks sampled around the timed region; per-stage times from a second
        graph with an event at every stage boundary (events serialise the
        kernels, so it is timed apart)."""
        for _ in range(max(3, warmup)):
            self.step()
        torch.cuda.synchronize()
        self.check()
        chunk = min(K, 256)
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(chunk)]
        for row in ev:          # torch creates the CUDA event on first record
            for e in row:
                e.record()
        torch.cuda.synchronize()
        stream = torch.cuda.Stream()
        stream.wait_stream(torch.cuda.current_stream())
        graphs = []
        with torch.cuda.stream(stream):
            for n in sorted({chunk, K % chunk} - {0}, reverse=True):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    for _ in range(n):
                        self.step()
                graphs.append((n, g))
            g_stages = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g_stages, stream=stream):
                for i in range(chunk):
                    self.step(ev[i])
        torch.cuda.current_stream().wait_stream(stream)
        plan = [graphs[0]] * (K // chunk) + ([g for g in graphs if g[0] == K % chunk] if K % chunk else [])
        for n, g in graphs:    # warm the graphs
            g.replay()
        g_stages.replay()
        torch.cuda.synchronize()
        clocks = ClockSampler(os.path.join(tempfile.gettempdir(), f"nvf_clocks_{os.getpid()}_{rank}.csv"))
        clocks.start()
        time.sleep(0.2)
        t_soak = time.perf_counter()
        while time.perf_counter() - t_soak < 1.0:
            plan[0][1].replay()
            torch.cuda.synchronize()
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        start.record()
        for n, g in plan:
            g.replay()
        end.record()
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        res = {"elapsed_ms": start.elapsed_time(end), "clocks": clocks.stop()}
        self.check()
        g_stages.replay()
        torch.cuda.synchronize()
        res["stage_ms"] = {s: statistics.mean(ev[i][a].elapsed_time(ev[i][b]) for i in range(chunk))
                           for s, a, b in STAGES}
        res["stage_step_ms"] = statistics.mean(ev[i][0].elapsed_time(ev[i][5]) for i in range(chunk))
        res["counts"] = self.counts()
        if e2e:
            # End to end through the C ABI with host buffers: every step copies x
            # and logits in from page-locked host memory, runs the layer and
            # copies out back.  Served as a decode engine would: the step is one
            # CUDA graph (nvf_moe_graph_create / _launch); the same step as
            # separate calls from Python (copies, nvfp4_moe_forward, copy) is
            # reported beside it.
            c = self.cfg
            g = self.nvf.MoEGraph(self.w, c.T, c.k, self.gs_a1, self.gs_a2, bias=self.bias,
                                  renormalize=c.renormalize, out_dtype=self.out.dtype)
            g.x.copy_(self.x.cpu())
            g.logits.copy_(self.logits.cpu())
            Ke = min(K, 200)
            for _ in range(3):
                g.launch()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(Ke):
                g.launch()
            e1.record()
            torch.cuda.synchronize()
            self.check()
            graph_ms = e0.elapsed_time(e1)
            g.close()
            xh, lh = self.x.cpu().pin_memory(), self.logits.cpu().pin_memory()
            oh = torch.empty(self.out.shape, dtype=self.out.dtype).pin_memory()
            xd, ld = torch.empty_like(self.x), torch.empty_like(self.logits)
            torch.cuda.synchronize()
            e0.record()
            for _ in range(Ke):
                xd.copy_(xh, non_blocking=True)
                ld.copy_(lh, non_blocking=True)
                self.step(x=xd, logits=ld)
                oh.copy_(self.out, non_blocking=True)
            e1.record()
            torch.cuda.synchronize()
            self.check()
            res.update(e2e_ms=graph_ms, e2e_eager_ms=e0.elapsed_time(e1), e2e_steps=Ke,
                       h2d=self.x.numel() * 2 + self.logits.numel() * 4, d2h=self.out.numel() * self.out.element_size())
        return res


def gemm_rooflines(cfg, t, touched, hbm, fp4_peak, src):
    """Per-GEMM rates from the stage times: algorithmic bytes (weights of the
    touched experts) and FLOPs, the fractions of the measured HBM copy rate and
    of the dense FP4 tensor peak, and the fraction of the roofline time
    max(FLOPs / FP4 peak, bytes / HBM rate)."""
    R = cfg.R
    out = {}
    for name, stage, nbytes, flops in (
            ("gate_up", "gate_up_gemm_swiglu_quant", gemm1_bytes(cfg, touched), 4.0 * R * cfg.H * cfg.I),
            ("down", "down_gemm", gemm2_bytes(cfg, touched), 2.0 * R * cfg.H * cfg.I)):
        sec = t["stage_ms"][stage] * 1e-3
        t_hbm = nbytes / (hbm * 1e9)
        t_tc = flops / (fp4_peak * 1e12)
        out[name] = {"us": sec * 1e6, "algorithmic_bytes": nbytes, "flops": flops,
                     "gbs": nbytes / sec / 1e9, "hbm_frac": nbytes / sec / 1e9 / hbm,
                     "tflops": flops / sec / 1e12, "tc_frac_fp4": flops / sec / 1e12 / fp4_peak,
                     "roofline_bound": "hbm" if t_hbm >= t_tc else "tensor",
                     "roofline_us": max(t_hbm, t_tc) * 1e6, "roofline_frac": max(t_hbm, t_tc) / sec}
    out["peaks"] = {"hbm_gbs": hbm, "fp4_tflops": fp4_peak,
                    "source": f"{src}: HBM copy rate; FP4 = bf16 GEMM burst x 6 (nominal dense ratio 13.5 / 2.25)"}
    return out


def prefill_object(nvf, w, seed, K, warmup, hbm, fp4_peak, src):
    """The prefill half of the metric: the same layer (same weights) at 4096
    tokens, timed like the headline; the gate_up GEMM's fraction of the dense
    FP4 tensor peak is its roofline."""
    cfg = CONFIGS["prefill"]
    run = LayerRun(nvf, cfg, w, seed)
    t = run.time(K, warmup, None, 0)
    ms = t["elapsed_ms"] / K
    touched, lbytes = layer_bytes(cfg, t["counts"])
    gemms = gemm_rooflines(cfg, t, touched, hbm, fp4_peak, src)
    g1 = gemms["gate_up"]
    obj = {"workload": workload_config(cfg, 1)["workload"], "T": cfg.T, "steps": K, "ms_per_step": ms,
           "value": cfg.T / (ms * 1e-3), "unit": "tokens/s", "stage_ms": t["stage_ms"],
           "stage_graph_ms_per_step": t["stage_step_ms"], "touched_experts": touched,
           "layer_flops": 6.0 * cfg.R * cfg.H * cfg.I,
           "layer_tflops": 6.0 * cfg.R * cfg.H * cfg.I / (ms * 1e-3) / 1e12,
           "layer_gbs": lbytes / (ms * 1e-3) / 1e9, "gemms": gemms,
           "roofline": {"kernel": "grouped_gemm_kernel<SWIGLU_QUANT> (gate_up)", "bound": "tensor",
                        "achieved": g1["tflops"], "peak": fp4_peak, "unit": "TFLOP/s", "frac": g1["tc_frac_fp4"],
                        "traffic": traffic_from_profiles(cfg.name), "roofline_bound": g1["roofline_bound"],
                        "roofline_frac": g1["roofline_frac"], "duration_us": g1["us"],
                        "peak_source": f"{src} bf16 GEMM burst x 6"},
           "clocks": t["clocks"], "gpu_launches": kernels_per_step(cfg.T) * K}
    del run
    return obj


def gemm_sources_sha():
    """sha256 (16 hex digits) of the GEMM kernel's sources: gemm.cu and the
    headers it includes, concatenated in this order."""
    from nvfp4_moe_grouped_router_gb300 import build as b
    import hashlib
    h = hashlib.sha256()
    for f in ("gemm.cu", "quant_block.cuh", "layout.cuh", "ptx.cuh", "internal.h"):
        h.update(open(os.path.join(b.CSRC, f), "rb").read())
    return h.hexdigest()[:16]


def traffic_from_profiles(name):
    p = os.path.join(ROOT, "profiles", "gemm_traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    h = gemm_sources_sha()
    e = d.get(name)
    if not e or e.get("gemm_sources_sha") != h:
        return None
    return e.get("bytes_per_launch")


if __name__ == "__main__":
    main()
