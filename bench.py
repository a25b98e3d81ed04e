#!/usr/bin/env python3
"""Benchmark of the NVFP4 MoE expert forward on GB300.

One step = one moe_forward (route, permute, quantize, L1 grouped GEMM + SwiGLU
+ NVFP4 requant, L2 grouped GEMM, combine) over one batch of T tokens of a
seeded synthetic workload, with weights and inputs resident in HBM. Prints one
JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload prefill]
  python bench.py --impl reference ...   # the CPU oracle on a bounded sample

Multi-GPU: one process per GPU (torchrun); every rank runs an independent
replica on its own tokens (the expert forward has no exchange step when the
weights are replicated), the result is max-over-ranks time, "weak" scaling.
"""
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "MoE layer TFLOP/s & tokens/s at 1 GB300; % of FP4 tensor peak / HBM BW"
FP4_OVER_BF16 = 13.5 / 2.25        # nominal dense FP4 / dense BF16 tensor rate
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
KERNELS_PER_STEP_FUSED = 4         # fused dispatch 1, L1 1, L2 1, combine 1 (static front too)


def kernels_per_step(T, k, fused):
    """Kernels of one moe_forward: the fused dispatch path (its quantize +
    scatter a second kernel above B.FRONT_FUSED_QUANTIZE_MAX_ROWS routed
    rows), else route 1, permute 1 (up to 1024 slots) or 3, quantize 3, L1 1,
    L2 1, combine 1."""
    from nvfp4_block_scaled_05_gb300 import binding as B
    if fused:
        return KERNELS_PER_STEP_FUSED + (1 if T * k > B.FRONT_FUSED_QUANTIZE_MAX_ROWS else 0)
    return 1 + (1 if T * k <= 1024 else 3) + 3 + 3


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="prefill",
                    choices=["tiny", "decode", "prefill", "skewed", "prefill_small", "decode_small", "prefill_med", "prefill_e32",
                             "skewed_small",
                             "dsv4_decode", "dsv4_prefill"])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--cpu-experts", type=int, default=8,
                    help="experts whose routed rows form the CPU-baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--front", default="dynamic", choices=["dynamic", "split", "static"],
                    help="dynamic (or split): moe_forward, gs_x computed every step (one fused "
                         "dispatch kernel when the tokens fit it, else route/permute/quantize "
                         "kernels); static: moe_forward_static (one fused front kernel, gs_x "
                         "pre-computed once)")
    ap.add_argument("--graph", action="store_true", help="replay the step as a captured CUDA graph")
    ap.add_argument("--gemm-mode", type=int, default=0, choices=[0, 1],
                    help="grouped-GEMM kernel: 0 one CTA per tile (default), 1 2-SM pairs (clusters of two CTAs "
                         "sharing one MMA) where N %% 256 == 0")
    ap.add_argument("--op", default="moe", choices=["moe", "qnorm_rope", "linear"],
                    help="moe: the expert forward (default); qnorm_rope: the fused RMS norm + RoPE + "
                         "NVFP4 quantization of attention-head rows; linear: the shared-expert NVFP4 "
                         "linear (activation quantization + GEMM). The last two: one GPU.")
    return ap.parse_args()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def rank_token_seed(seed, rank):
    """Seed of the tokens (x, router logits) a rank processes: every rank runs
    an independent replica of the layer on its own batch (same weights, seed
    `seed`), so the work per rank is fixed as ranks are added (weak scaling)."""
    return seed if rank == 0 else seed + 7919 * rank


def max_over_ranks(values, pg, device):
    """Elementwise maximum of per-rank timings (list of floats) over all ranks."""
    import torch
    if pg is None:
        return list(values)
    t = torch.tensor(values, dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return t.tolist()


def aggregate_throughput(per_rank_flops, per_rank_tokens, world, ms):
    """Whole-job TFLOP/s and tokens/s: all ranks' work over the slowest rank's time."""
    return world * per_rank_flops / (ms * 1e-3) / 1e12, world * per_rank_tokens / (ms * 1e-3)


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples (every 200 ms) of SM clock and throttle reasons."""

    FIELDS = ["timestamp", "clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + ",".join(self.FIELDS),
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self, t_start=None, t_end=None):
        """Summary of the samples taken between t_start and t_end (time.time())."""
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) != len(self.FIELDS):
                    continue
                try:
                    ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                except ValueError:
                    continue
                if (t_start is None or ts >= t_start) and (t_end is None or ts <= t_end):
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(v):
            try:
                return float(v)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        pw = [num(r[3]) for r in rows if num(r[3]) is not None]
        load = sm
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for n, v in zip(names, r[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(load or sm) if (load or sm) else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(rows), "samples_under_load": len(load)}


# ---------------------------------------------------------------- helpers

def kernel_source_hash():
    h = hashlib.sha256()
    for f in ["gemm.cu", "common.cuh"]:
        with open(os.path.join(ROOT, "nvfp4_block_scaled_05_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(workload):
    """dram bytes per launch of the L1 kernel from the committed ncu summary,
    or None when the summary was taken on other kernel sources."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    if not os.path.exists(path):
        return None
    src = kernel_source_hash()
    with open(path) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            kv = dict(p.split("=", 1) for p in line.split() if "=" in p)
            if kv.get("workload") == workload and kv.get("kernel") == "l1_swiglu" and \
                    kv.get("source") == src:
                return float(kv["dram_bytes_per_launch"])
    return None


def layer_numbers(cfg, offsets):
    """Algorithmic FLOPs and bytes of one forward and of the L1 kernel.

    The L1 kernel's algorithmic bytes are its active experts' W1 codes and
    scales only; the activation rows it reads (A) and the h rows it writes are
    pipeline bytes between kernels, reported apart (l1_pipeline_bytes)."""
    counts = [offsets[e + 1] - offsets[e] for e in range(cfg.E)]
    active = sum(1 for c in counts if c > 0)
    K, I, M, T = cfg.K, cfg.I, cfg.M, cfg.T
    w1 = 2 * I * (K // 2 + K // 16)
    w2 = K * (I // 2 + I // 16)
    flops = 6.0 * M * K * I
    layer_bytes = active * (w1 + w2) + T * K * 2 * 2 + T * cfg.E * 4
    l1_flops = 4.0 * M * K * I
    l1_bytes = active * w1
    l1_pipeline = M * (K // 2 + K // 16) + M * (I // 2 + I // 16)
    return dict(active=active, flops=flops, bytes=layer_bytes, l1_flops=l1_flops, l1_bytes=l1_bytes,
                l1_pipeline_bytes=l1_pipeline)


def l1_roofline(nums, l1_ms, hbm_peak, fp4_peak):
    """Roofline of the L1 kernel: bound by W1 streaming (HBM) or by the FP4
    tensor rate, whichever takes longer at the peaks; achieved = algorithmic
    bytes (or FLOPs) over the kernel's measured time."""
    t_hbm = nums["l1_bytes"] / (hbm_peak * 1e9)
    t_tc = nums["l1_flops"] / (fp4_peak * 1e12)
    if t_hbm >= t_tc:
        achieved = nums["l1_bytes"] / (l1_ms * 1e-3) / 1e9
        return {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                "frac": achieved / hbm_peak}
    achieved = nums["l1_flops"] / (l1_ms * 1e-3) / 1e12
    return {"bound": "tensor", "achieved": achieved, "peak": fp4_peak, "unit": "TFLOP/s",
            "frac": achieved / fp4_peak}


# ---------------------------------------------------------------- oracle legs

_HOST_INPUTS = {}


def oracle_sample(cfg, seed, n_experts, step=0):
    """Host inputs of a bounded sample: all routed rows of n_experts experts.
    Inputs are drawn on the CPU (same distributions as the GPU workload)."""
    import numpy as np
    import oracle as O
    from nvfp4_block_scaled_05_gb300 import workloads as W
    key = (cfg.name, seed)
    if key not in _HOST_INPUTS:
        inp = W.moe_inputs(cfg, seed=seed, device="cpu", weights=False)
        lg = inp["logits"].numpy()
        _HOST_INPUTS[key] = (W.bf16_bits(inp["x"]), lg, O.route_topk(lg, cfg.k)[0])
    x, logits, ids = _HOST_INPUTS[key]
    counts = np.bincount(ids.ravel(), minlength=cfg.E)
    active = [e for e in range(cfg.E) if counts[e] > 0]
    experts = [active[(step * n_experts + i) % len(active)] for i in range(n_experts)]
    qw = {}
    for e in experts:
        c1, s1, g1 = O.quantize_expert(W.bf16_bits(W.expert_weight(cfg, seed, 1, e)))
        c2, s2, g2 = O.quantize_expert(W.bf16_bits(W.expert_weight(cfg, seed, 2, e)))
        qw[e] = (c1, s1, g1, c2, s2, g2)
    tokens = sorted(set(int(t) for t, j in zip(*np.nonzero(np.isin(ids, experts)))))
    rows = int(np.isin(ids, experts).sum())
    return dict(x=x, logits=logits, experts=experts, qw=qw, tokens=tokens, rows=rows)


def time_oracle(cfg, sample):
    import numpy as np
    import oracle as O
    t0 = time.perf_counter()
    O.moe_forward(sample["x"], sample["logits"], None, None, cfg.k, np.float32(cfg.gs_h),
                  tokens=sample["tokens"], experts=set(sample["experts"]),
                  qweights=lambda e: sample["qw"][e])
    dt = time.perf_counter() - t0
    flops = 6.0 * cfg.K * cfg.I * sample["rows"]
    return dt, flops


def full_size_parity(cfg, seed, n_experts, x, logits, dev, f2p, out, topk_w, max_rows=None):
    """Parity of the benchmarked run itself on a bounded sample: for every token
    routed to one of n_experts active experts, those experts' share of y,
    sum_j w[t,j] * out[t,j] over the slots j routed to them, formed from the
    L2 output rows and routing weights left in the workspace by the last timed
    forward, against the oracle's fp64 share on the same inputs (x and logits
    copied back, the sampled experts' weights drawn again on the device: the
    same values as the run's), with the layer tolerance (2e-2 * max(1, |y|)).
    max_rows: only experts with at most that many routed rows are sampled (the
    first n_experts of them in index order), which bounds the oracle's time."""
    import numpy as np
    import oracle as O
    from nvfp4_block_scaled_05_gb300 import workloads as W
    xb = W.bf16_bits(x.cpu())
    lg = logits.cpu().numpy()
    ids = O.route_topk(lg, cfg.k)[0]
    counts = np.bincount(ids.ravel(), minlength=cfg.E)
    experts = [e for e in range(cfg.E) if counts[e] > 0 and (max_rows is None or counts[e] <= max_rows)]
    experts = experts[:n_experts]
    qw = {}
    for e in experts:
        c1, s1, g1 = O.quantize_expert(W.bf16_bits(W.expert_weight(cfg, seed, 1, e, dev).cpu()))
        c2, s2, g2 = O.quantize_expert(W.bf16_bits(W.expert_weight(cfg, seed, 2, e, dev).cpu()))
        qw[e] = (c1, s1, g1, c2, s2, g2)
    tokens = sorted(set(int(t) for t, j in zip(*np.nonzero(np.isin(ids, experts)))))
    t0 = time.perf_counter()
    ref = O.moe_forward(xb, lg, None, None, cfg.k, np.float32(cfg.gs_h), tokens=tokens, experts=set(experts),
                        qweights=lambda e: qw[e], keep=True)
    dt = time.perf_counter() - t0
    tix = {t: i for i, t in enumerate(ref["tokens"])}
    share = np.zeros((len(tix), cfg.K), np.float64)
    rows_got, rows_want = [], []
    for (t, j), d in ref["inter"].items():
        row = (out[f2p[t * cfg.k + j]].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        share[tix[t]] += float(topk_w[t * cfg.k + j]) * row
        rows_got.append(row)
        rows_want.append(d["o"])
    want = ref["y"]
    err = np.abs(share - want) / np.maximum(1.0, np.abs(want))
    cos = float((share * want).sum() / np.sqrt((share * share).sum() * (want * want).sum()))
    rg, rw = np.array(rows_got), np.array(rows_want)
    rcos = float((rg * rw).sum() / np.sqrt((rg * rg).sum() * (rw * rw).sum()))
    parity = {"tokens": len(tix), "routed_rows": len(rows_got), "experts": experts,
              "max_err_over_tol": float(err.max()), "tolerance": 2e-2, "within": bool(err.max() <= 2e-2),
              "cosine": cos, "l2_rows_cosine": rcos,
              "compared": "the sampled experts' share of y for every token routed to them, formed from the "
                          "benchmarked run's L2 output rows and routing weights, against the fp64 oracle on "
                          "the same inputs"}
    flops = 6.0 * cfg.K * cfg.I * len(rows_got)
    cpu = {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": O.get_threads(), "kind": "oracle",
           "sample": "all %d routed rows of %d experts (%s) of this run's inputs, routing and global scale over "
                     "all %d tokens; weights quantized beforehand; %.1f s"
                     % (len(rows_got), len(experts), ",".join(map(str, experts)), cfg.T, dt)}
    return parity, cpu


_QW_CACHE = {}


def oracle_step_sample(cfg, seed, step, max_rows, n_experts=4):
    """One step of the reference arm: the tokens routed to one of the first
    n_experts active experts (cycled by step), at most max_rows of them (None:
    all). The experts' quantized weights are drawn once and kept, so a step
    costs only the oracle's arithmetic."""
    import numpy as np
    import oracle as O
    from nvfp4_block_scaled_05_gb300 import workloads as W
    key = (cfg.name, seed)
    if key not in _HOST_INPUTS:
        inp = W.moe_inputs(cfg, seed=seed, device="cpu", weights=False)
        lg = inp["logits"].numpy()
        _HOST_INPUTS[key] = (W.bf16_bits(inp["x"]), lg, O.route_topk(lg, cfg.k)[0])
    x, logits, ids = _HOST_INPUTS[key]
    counts = np.bincount(ids.ravel(), minlength=cfg.E)
    active = [e for e in range(cfg.E) if counts[e] > 0]
    e = active[step % min(n_experts, len(active))]
    if (key, e) not in _QW_CACHE:
        c1, s1, g1 = O.quantize_expert(W.bf16_bits(W.expert_weight(cfg, seed, 1, e)))
        c2, s2, g2 = O.quantize_expert(W.bf16_bits(W.expert_weight(cfg, seed, 2, e)))
        _QW_CACHE[(key, e)] = (c1, s1, g1, c2, s2, g2)
    tokens = sorted(set(int(t) for t in np.nonzero((ids == e).any(axis=1))[0]))
    if max_rows is not None:
        tokens = tokens[:max_rows]
    return dict(x=x, logits=logits, experts=[e], qw={e: _QW_CACHE[(key, e)]}, tokens=tokens,
                rows=len(tokens))


def run_reference(args, cfg):
    """The CPU oracle, timed on the host cores, on a bounded sample of the
    workload: every step runs the routed rows of one expert (cycling over four
    experts whose weights are prepared once), with the rows per step chosen
    from two calibration calls so that all warm-up and timed steps together
    take about two and a half minutes (longer only when the per-call cost
    alone exceeds that: one row per step then)."""
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle as O
    # calibration: a one-row call (the per-call cost: routing, permutation and
    # global scale over all tokens, the expert's weights dequantized) and a
    # whole-expert call (the cost per row)
    one = oracle_step_sample(cfg, args.seed, 0, 1)
    fixed, _ = time_oracle(cfg, one)
    calib = oracle_step_sample(cfg, args.seed, 0, None)
    dt0, _ = time_oracle(cfg, calib)
    per_row = max(dt0 - fixed, 1e-6) / max(1, calib["rows"] - 1)
    n_total = max(1, args.warmup + args.steps)
    budget = 150.0 / n_total - fixed      # seconds of row work per step
    max_rows = max(1, min(calib["rows"], int(budget / per_row) if budget > 0 else 1))
    for i in range(args.warmup):
        time_oracle(cfg, oracle_step_sample(cfg, args.seed, i, max_rows))
    total_t, total_f, rows = 0.0, 0.0, 0
    for i in range(args.steps):
        s = oracle_step_sample(cfg, args.seed, args.warmup + i, max_rows)
        dt, fl = time_oracle(cfg, s)
        total_t += dt
        total_f += fl
        rows += s["rows"]
    value = total_f / total_t / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": total_t / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64 (oracle)", "data": "synthetic",
            "config": {"workload": cfg.name, "T": cfg.T, "K": cfg.K, "I": cfg.I, "E": cfg.E, "k": cfg.k,
                       "seed": args.seed,
                       "step": "up to %d routed rows of one expert (of 4, cycled) per step" % max_rows},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": O.get_threads(),
                             "kind": "oracle",
                             "sample": "%d steps x up to %d routed rows of one expert (%d rows in total)"
                                       % (args.steps, max_rows, rows)},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- GPU leg

def run_ours(args, cfg):
    import torch
    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist
    from nvfp4_block_scaled_05_gb300 import binding as B
    from nvfp4_block_scaled_05_gb300 import workloads as W
    B.nvfp4moe_set_gemm_mode(args.gemm_mode)

    # inputs: replicated weights (same seed on every rank), per-rank tokens
    inp = W.moe_inputs(cfg, seed=args.seed, device=dev, weights=True)
    if rank:
        tok = W.moe_inputs(cfg, seed=rank_token_seed(args.seed, rank), device=dev, weights=False)
        inp["x"], inp["logits"] = tok["x"], tok["logits"]
    wts = B.prepare_moe_weights(inp["w1"], inp["w2"])
    del inp["w1"], inp["w2"]
    torch.cuda.empty_cache()
    x, logits = inp["x"], inp["logits"]
    gs_h = torch.tensor([cfg.gs_h], dtype=torch.float32, device=dev)
    T, K, I, E, k = cfg.T, cfg.K, cfg.I, cfg.E, cfg.k
    ws = torch.empty(B.moe_forward_workspace_size(T, K, I, E, k), dtype=torch.uint8, device=dev)
    y = torch.empty((T, K), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream()

    def barrier():
        torch.cuda.synchronize()
        if pg is not None:
            pg.barrier()

    static = args.front == "static"
    gs_x = None
    if static:
        # the pre-computed activation scale: one calibration forward's gs_x
        B.moe_forward(x, logits, wts, k, gs_h, ws=ws, y=y)
        lay0 = B.moe_forward_workspace_layout(T, K, I, E, k)
        gs_x = ws[lay0["gs_x"]:lay0["gs_x"] + 4].view(torch.float32).clone()

    def forward_into(xx, ll, yy):
        if static:
            B.moe_forward_static(xx, ll, wts, k, gs_h, gs_x, ws=ws, y=yy)
        else:
            B.moe_forward(xx, ll, wts, k, gs_h, ws=ws, y=yy)

    def forward(xx, ll):
        forward_into(xx, ll, y)

    def captured(xx, ll):
        """forward(xx, ll) as a replayable CUDA graph (or None without --graph)."""
        if not args.graph:
            return None
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            forward(xx, ll)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side):
                forward(xx, ll)
        stream.wait_stream(side)
        torch.cuda.synchronize()
        return g

    # ---- device-resident timing of the forward
    graph = captured(x, logits)
    run = graph.replay if graph is not None else (lambda: forward(x, logits))
    for _ in range(args.warmup):
        run()
    st = B.nvfp4moe_last_device_status()
    if st != 0:
        raise RuntimeError("device status %d after warm-up" % st)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(1.0)                      # let the sampler start before the timed region
    barrier()
    t_start = time.time()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(args.steps):
        run()
    ev1.record(stream)
    barrier()
    t_end = time.time()
    clk = clocks.stop(t_start, t_end)
    ms = ev0.elapsed_time(ev1) / args.steps
    if B.nvfp4moe_last_device_status() != 0:
        raise RuntimeError("device status after timed region")

    # ---- per-stage device time (same stream, events between the six calls)
    fused_front = static or B.moe_forward_uses_fused_dispatch(T, E, k)
    names = B.STATIC_STAGES if static else B.forward_stages(T, E, k)
    nst = len(names)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(nst + 1)] for _ in range(args.steps)]
    barrier()
    for i in range(args.steps):
        if static:
            B.moe_forward_static_stages(x, logits, wts, k, gs_h, gs_x, ws, y, events=evs[i])
        else:
            B.moe_forward_stages(x, logits, wts, k, gs_h, ws, y, events=evs[i])
    barrier()
    stage_ms = {name: sum(evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(args.steps)) / args.steps
                for j, name in enumerate(names)}

    # ---- end to end through the public call, host buffers, copies timed.
    # Every step copies its own inputs from pinned host memory and its output
    # back; copies run on their own streams, double-buffered, so step i's
    # copies overlap the neighbouring steps' compute (a serving pipeline).
    x_h = x.cpu().pin_memory()
    l_h = logits.cpu().pin_memory()
    y_h = [torch.empty((T, K), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    x_d = [torch.empty_like(x) for _ in range(2)]
    l_d = [torch.empty_like(logits) for _ in range(2)]
    y_d = [torch.empty_like(y) for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    graphs_e2e = [None, None]
    if args.graph:
        for j in range(2):
            side = torch.cuda.Stream()
            side.wait_stream(stream)
            with torch.cuda.stream(side):
                forward_into(x_d[j], l_d[j], y_d[j])
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=side):
                    forward_into(x_d[j], l_d[j], y_d[j])
            stream.wait_stream(side)
            graphs_e2e[j] = g
        torch.cuda.synchronize()
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def pipelined(nsteps):
        for i in range(nsteps):
            j = i & 1
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(ev_done[j])          # buffers j free once step i-2 computed
                x_d[j].copy_(x_h, non_blocking=True)
                l_d[j].copy_(l_h, non_blocking=True)
                ev_in[j].record(s_in)
            stream.wait_event(ev_in[j])
            if i >= 2:
                stream.wait_event(ev_out[j])             # y_d[j] read back by step i-2
            if graphs_e2e[j] is not None:
                graphs_e2e[j].replay()
            else:
                forward_into(x_d[j], l_d[j], y_d[j])
            ev_done[j].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_done[j])
                y_h[j].copy_(y_d[j], non_blocking=True)
                ev_out[j].record(s_out)

    pipelined(max(2, args.warmup // 2))
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    pipelined(args.steps)
    stream.wait_stream(s_out)
    e1.record(stream)
    barrier()
    e2e_ms = e0.elapsed_time(e1) / args.steps
    if not torch.equal(y_h[(args.steps - 1) & 1], y.cpu()):
        raise RuntimeError("end-to-end output differs from the device-resident run")

    lay = B.moe_forward_workspace_layout(T, K, I, E, k)
    offsets = ws[lay["offsets"]:lay["offsets"] + 4 * (E + 1)].view(torch.int32).cpu().tolist()
    nums = layer_numbers(cfg, offsets)

    ms, e2e_ms, l1_ms = max_over_ranks([ms, e2e_ms, stage_ms["l1_swiglu"]], pg, dev)
    if rank != 0:
        if pg is not None:
            pg.barrier()
            pg.destroy_process_group()
        return

    peaks, peak_kind = load_peaks()
    hbm_peak = float(peaks["hbm_gbs"])
    fp4_peak = float(peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"])) * FP4_OVER_BF16
    tflops, tokens_s = aggregate_throughput(nums["flops"], T, world, ms)
    # roofline of the dominant kernel (L1 grouped GEMM + SwiGLU + requant)
    roof = l1_roofline(nums, l1_ms, hbm_peak, fp4_peak)
    roof["algorithmic"] = ("active experts x W1 codes and scales (%d x %d B)" %
                           (nums["active"], 2 * I * (K // 2 + K // 16)) if roof["bound"] == "hbm" else
                           "4*M*K*I FLOP")
    roof["traffic"] = ncu_traffic(cfg.name)
    roof["l1_pipeline_bytes"] = nums["l1_pipeline_bytes"]
    roof["kernel"] = "l1_swiglu (grouped_gemm_kernel<true>)"
    roof["kernel_ms"] = l1_ms
    roof["peak_source"] = "%s (MEASURED_PEAKS.json)" % peak_kind if peak_kind == "measured" else "fallback"
    if roof["bound"] == "tensor":
        roof["peak_note"] = "measured sustained bf16 x 6 (nominal dense fp4/bf16 ratio)"
    line = {
        "metric": METRIC, "value": tflops, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "nvfp4 (e2m1 x e4m3 block scale, f32 accumulate)",
        "data": "synthetic (seeded; random-init weights of the layer shape)",
        "config": {"workload": cfg.name, "T": T, "K": K, "I": I, "E": E, "k": k, "M": cfg.M,
                   "global_tokens": world * T, "parallelism": "replicas x%d" % world,
                   "active_experts": nums["active"], "seed": args.seed, "gs_h": cfg.gs_h,
                   "front": ("static (moe_forward_static; gs_x pre-computed once by a calibration "
                             "forward)" if static else
                             (("fused dispatch kernel (gs_x computed every step)"
                               if T * k <= B.FRONT_FUSED_QUANTIZE_MAX_ROWS else
                               "fused routing + permutation kernel, then the quantize + scatter kernel "
                               "(gs_x computed every step)") if fused_front else
                              "route, permute and quantize kernels (gs_x computed every step)")),
                   "cuda_graph": bool(args.graph),
                   "gemm_kernel": "2-SM pairs" if args.gemm_mode == 1 else "one CTA per tile",
                   "l2": "inputs larger than L2: %.2f GB of expert weights streamed every step"
                         % (nums["bytes"] / 1e9)},
        "tokens_per_s": tokens_s,
        "pct_fp4_peak": tflops / world / fp4_peak,
        "pct_hbm_bw": nums["bytes"] / (ms * 1e-3) / 1e9 / hbm_peak,
        # the layer against its own roofline: the larger of the two bounds over the time
        "layer_roofline_frac": max(tflops / world / fp4_peak, nums["bytes"] / (ms * 1e-3) / 1e9 / hbm_peak),
        # bytes of the intermediates between the kernels, reported apart from the
        # algorithmic bytes (A in FP4 + scales, h in FP4 + scales, L2 output written and
        # read back by the combine)
        "pipeline_bytes": {"a_fp4": cfg.M * (K // 2 + K // 16), "h_fp4": cfg.M * (I // 2 + I // 16),
                           "l2_out_bf16": 2 * cfg.M * K * 2},
        "layer_bytes": nums["bytes"], "layer_flops": nums["flops"],
        "stages_ms": stage_ms,
        "roofline": roof,
        "e2e": {"value": world * nums["flops"] / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                "ms_per_step": e2e_ms, "h2d_bytes_per_step": x.numel() * 2 + logits.numel() * 4,
                "d2h_bytes_per_step": y.numel() * 2,
                "copies": "pinned host <-> device every step, on their own streams, double-buffered "
                          "(overlapping the neighbouring steps' compute)"},
        "gpu_launches": kernels_per_step(T, k, fused_front) * args.steps,
        "clocks": clk,
    }
    if world == 1 and cfg.name == "prefill" and not args.graph and not static:
        # the other two layer targets (decode: HBM; skewed: FP4 tensor rate) on the same weights
        line["also"] = measure_also(args, cfg, wts, dev, hbm_peak, fp4_peak)
        line["gpu_launches_also"] = sum(kernels_per_step(W.CONFIGS[n].T, W.CONFIGS[n].k,
                                                         B.moe_forward_uses_fused_dispatch(
                                                             W.CONFIGS[n].T, W.CONFIGS[n].E, W.CONFIGS[n].k))
                                        * v["steps"] for n, v in line["also"].items())
    if world == 1 and not args.no_cpu_baseline:
        M = cfg.M
        f2p_h = ws[lay["flat_to_perm"]:lay["flat_to_perm"] + 4 * M].view(torch.int32).cpu().numpy()
        out_h = ws[lay["out"]:lay["out"] + 2 * M * K].view(torch.int16).view(M, K).cpu().numpy().view("uint16")
        tw_h = ws[lay["topk_w"]:lay["topk_w"] + 4 * M].view(torch.float32).cpu().numpy()
        line["parity"], line["cpu_baseline"] = full_size_parity(cfg, args.seed, args.cpu_experts, x, logits, dev,
                                                               f2p_h, out_h, tw_h)
    print(json.dumps(line), flush=True)
    if pg is not None:
        pg.barrier()
        pg.destroy_process_group()


def measure_also(args, base, wts, dev, hbm_peak, fp4_peak):
    """The decode (T=128) and skewed (T=16384) workloads, measured in the same
    run on the benchmarked layer's weights (all three workloads share K, I, E
    and the weight seed, so the weights are the same tensors). Per workload:
    ms per step over timed moe_forward calls (CUDA events, after warm-up; the
    6.3 GB of weights streamed every step exceed L2), TFLOP/s, tokens/s,
    % of HBM bandwidth and of the FP4 peak, and the L1 kernel's roofline
    fraction from its own per-stage time."""
    import torch
    from nvfp4_block_scaled_05_gb300 import binding as B
    from nvfp4_block_scaled_05_gb300 import workloads as W
    out = {}
    stream = torch.cuda.current_stream()
    for name in ("decode", "skewed"):
        cfg = W.CONFIGS[name]
        if (cfg.K, cfg.I, cfg.E) != (base.K, base.I, base.E):
            continue
        inp = W.moe_inputs(cfg, seed=args.seed, device=dev, weights=False)
        x, logits = inp["x"], inp["logits"]
        T, K, I, E, k = cfg.T, cfg.K, cfg.I, cfg.E, cfg.k
        ws = torch.empty(B.moe_forward_workspace_size(T, K, I, E, k), dtype=torch.uint8, device=dev)
        y = torch.empty((T, K), dtype=torch.bfloat16, device=dev)
        gs_h = torch.tensor([cfg.gs_h], dtype=torch.float32, device=dev)
        steps = max(20, args.steps if name == "decode" else args.steps // 4)
        for _ in range(max(3, args.warmup)):
            B.moe_forward(x, logits, wts, k, gs_h, ws=ws, y=y)
        torch.cuda.synchronize()
        if B.nvfp4moe_last_device_status() != 0:
            raise RuntimeError("device status after warm-up (%s)" % name)
        clocks = ClockSampler(torch.cuda.current_device())
        clocks.start()
        time.sleep(0.6)
        t0 = time.time()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            B.moe_forward(x, logits, wts, k, gs_h, ws=ws, y=y)
        e1.record(stream)
        torch.cuda.synchronize()
        clk = clocks.stop(t0, time.time())
        ms = e0.elapsed_time(e1) / steps
        names = B.forward_stages(T, E, k)
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1)] for _ in range(steps)]
        for i in range(steps):
            B.moe_forward_stages(x, logits, wts, k, gs_h, ws, y, events=evs[i])
        torch.cuda.synchronize()
        if B.nvfp4moe_last_device_status() != 0:
            raise RuntimeError("device status after timed region (%s)" % name)
        stage_ms = {n: sum(evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(steps)) / steps
                    for j, n in enumerate(names)}
        lay = B.moe_forward_workspace_layout(T, K, I, E, k)
        offsets = ws[lay["offsets"]:lay["offsets"] + 4 * (E + 1)].view(torch.int32).cpu().tolist()
        parity = None
        if not args.no_cpu_baseline:
            # the last forward's L2 rows and routing against the oracle, as for
            # the benchmarked workload (a bounded sample of experts)
            M = T * k
            f2p_h = ws[lay["flat_to_perm"]:lay["flat_to_perm"] + 4 * M].view(torch.int32).cpu().numpy()
            out_h = ws[lay["out"]:lay["out"] + 2 * M * K].view(torch.int16).view(M, K).cpu().numpy().view("uint16")
            tw_h = ws[lay["topk_w"]:lay["topk_w"] + 4 * M].view(torch.float32).cpu().numpy()
            parity, _ = full_size_parity(cfg, args.seed, 8 if name == "decode" else 4, x, logits, dev,
                                         f2p_h, out_h, tw_h, max_rows=None if name == "decode" else 600)
        nums = layer_numbers(cfg, offsets)
        roof = l1_roofline(nums, stage_ms["l1_swiglu"], hbm_peak, fp4_peak)
        tf = nums["flops"] / (ms * 1e-3) / 1e12
        out[name] = {"T": T, "steps": steps, "ms_per_step": ms, "tflops": tf, "tokens_per_s": T / (ms * 1e-3),
                     "pct_hbm_bw": nums["bytes"] / (ms * 1e-3) / 1e9 / hbm_peak, "pct_fp4_peak": tf / fp4_peak,
                     "active_experts": nums["active"], "stages_ms": stage_ms,
                     "l1_roofline": {"bound": roof["bound"], "frac": roof["frac"], "achieved": roof["achieved"],
                                     "unit": roof["unit"], "kernel_ms": stage_ms["l1_swiglu"],
                                     "traffic": ncu_traffic(name)},
                     "clocks": clk}
        if parity is not None:
            out[name]["parity"] = parity
        del ws, y, x, logits
        torch.cuda.empty_cache()
    return out


# ---------------------------------------------------------------- side ops

def _timed(stream, steps, fn, flush=None, min_seconds=0.0):
    """Device ms per call of fn(): CUDA events on `stream` around each call; an
    optional flush() runs outside the timed spans. At least `steps` calls, and
    more until `min_seconds` of wall time passed (so the clock sampler sees the
    timed region). Returns (ms per call, calls)."""
    import torch
    total, n = 0.0, 0
    t0 = time.time()
    while n < steps or time.time() - t0 < min_seconds:
        if flush is not None:
            flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        b.synchronize()
        total += a.elapsed_time(b)
        n += 1
    return total / n, n


def _side_line(args, metric, value, unit, ms, config, roof, e2e, launches, clk, cpu, steps):
    return {"metric": metric, "value": value, "unit": unit, "n_gpus": 1, "steps": steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "nvfp4 out (e2m1 x e4m3 block scale), f32 arithmetic",
            "data": "synthetic (seeded)", "config": config, "roofline": roof, "e2e": e2e,
            "gpu_launches": launches, "clocks": clk, "cpu_baseline": cpu}


def run_qnorm_rope(args):
    """RMS norm -> RoPE -> NVFP4 of q-head rows: T=8192 tokens x 128 heads, head
    dim 192 (128 plain + 64 rotary), positions = token index, standard RoPE
    frequencies (base 10000) as f32 tables, pre-computed global scale."""
    import numpy as np
    import torch
    from nvfp4_block_scaled_05_gb300 import binding as B
    dev = torch.device("cuda", 0)
    T, H, D, R = 8192, 128, 192, 64
    rows = T * H
    g = torch.Generator(device=dev).manual_seed(args.seed)
    x = torch.randn(rows, D, generator=g, device=dev).to(torch.bfloat16)
    gamma = (1.0 + 0.1 * torch.randn(D, generator=g, device=dev)).float()
    inv = 10000.0 ** (-torch.arange(0, R, 2, dtype=torch.float64) / R)
    ang = torch.arange(T, dtype=torch.float64)[:, None] * inv[None, :]
    cos_t, sin_t = torch.cos(ang).float().to(dev), torch.sin(ang).float().to(dev)
    pos = torch.arange(T, dtype=torch.int32, device=dev).repeat_interleave(H)
    codes = torch.empty((rows, D // 2), dtype=torch.uint8, device=dev)
    sf = torch.empty(B.nvfp4_sf_bytes(rows, D), dtype=torch.uint8, device=dev)
    one = torch.ones(1, device=dev)
    y = torch.empty((rows, D), dtype=torch.float32, device=dev)
    B.nvfp4_rmsnorm_rope_quantize(x, gamma, 1e-6, R, pos, cos_t, sin_t, one, y_out=y, codes=codes, sf=sf)
    gs = torch.tensor([2688.0 / y.abs().max().item()], device=dev)     # calibration: the pre-computed scale
    del y
    stream = torch.cuda.current_stream()
    fn = lambda: B.nvfp4_rmsnorm_rope_quantize(x, gamma, 1e-6, R, pos, cos_t, sin_t, gs, codes=codes, sf=sf)
    for _ in range(args.warmup):
        fn()
    torch.cuda.synchronize()
    if B.nvfp4moe_last_device_status() != 0:
        raise RuntimeError("device status after warm-up")
    clocks = ClockSampler(0)
    clocks.start()
    time.sleep(1.0)
    t0 = time.time()
    ms, steps = _timed(stream, args.steps, fn, min_seconds=1.5)   # inputs (403 MB) exceed L2
    clk = clocks.stop(t0, time.time())
    per_row = 2 * D + 4 + D // 2 + D // 16
    alg = rows * per_row
    gbs = alg / (ms * 1e-3) / 1e9
    peaks, kind = load_peaks()
    hbm = float(peaks["hbm_gbs"])
    # end to end: x and positions from pinned host memory, codes and scales back
    x_h, p_h = x.cpu().pin_memory(), pos.cpu().pin_memory()
    c_h = torch.empty(codes.shape, dtype=torch.uint8).pin_memory()
    s_h = torch.empty(sf.shape, dtype=torch.uint8).pin_memory()
    x_d, p_d = torch.empty_like(x), torch.empty_like(pos)

    def e2e_step():
        x_d.copy_(x_h, non_blocking=True)
        p_d.copy_(p_h, non_blocking=True)
        B.nvfp4_rmsnorm_rope_quantize(x_d, gamma, 1e-6, R, p_d, cos_t, sin_t, gs, codes=codes, sf=sf)
        c_h.copy_(codes, non_blocking=True)
        s_h.copy_(sf, non_blocking=True)
    e2e_step()
    e2e_ms, _ = _timed(stream, max(3, args.steps // 10), e2e_step)
    # CPU oracle on a bounded sample of the same rows
    import oracle as O
    from nvfp4_block_scaled_05_gb300 import workloads as W
    n = 16384
    xs = W.bf16_bits(x[:n].cpu())
    c0 = time.perf_counter()
    yo = O.rmsnorm_rope(xs, gamma.double().cpu().numpy(), 1e-6, R, pos[:n].cpu().numpy(),
                        cos_t.double().cpu().numpy(), sin_t.double().cpu().numpy())
    O.quantize_f32(yo.astype(np.float32), np.float32(gs.item()))
    dt = time.perf_counter() - c0
    cpu = {"value": n * per_row / dt / 1e9, "unit": "GB/s", "cores": O.get_threads(), "kind": "oracle",
           "sample": "%d of the %d rows (norm + rope in fp64, then the f32 quantizer); %.1f s" % (n, rows, dt)}
    line = _side_line(
        args, "fused RMS norm + RoPE + NVFP4 quant of q-head rows, algorithmic GB/s", gbs, "GB/s", ms,
        {"workload": "qnorm_rope", "tokens": T, "heads": H, "head_dim": D, "rope_dims": R, "rows": rows,
         "l2": "inputs larger than L2 (403 MB of BF16 rows)", "bytes_per_row": per_row},
        {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": gbs / hbm, "traffic": None,
         "kernel": "norm_rope_quantize_kernel", "kernel_ms": ms, "peak_source": kind},
        {"value": alg / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s", "ms_per_step": e2e_ms,
         "h2d_bytes_per_step": x.numel() * 2 + pos.numel() * 4,
         "d2h_bytes_per_step": codes.numel() + sf.numel()},
        steps, clk, cpu, steps)
    print(json.dumps(line), flush=True)


def run_linear(args):
    """The shared-expert linear (M=4096, K=7168, N=4096): dynamic-gs NVFP4
    quantization of the BF16 activation, then nvfp4_linear to BF16."""
    import numpy as np
    import torch
    from nvfp4_block_scaled_05_gb300 import binding as B
    from nvfp4_block_scaled_05_gb300 import workloads as W
    dev = torch.device("cuda", 0)
    cfg = W.CONFIGS["linear"]
    inp = W.linear_inputs(cfg, seed=args.seed, device=dev)
    M, K, N = cfg.M, cfg.K, cfg.N
    x = inp["x"]
    wc, wsf, gsw = B.nvfp4_quantize(inp["w"][0])
    a_rows = -(-M // 128) * 128
    xc = torch.zeros((a_rows, K // 2), dtype=torch.uint8, device=dev)
    xsf = torch.zeros(B.nvfp4_sf_bytes(a_rows, K, B.NVFP4_SF_TILED_ROWS), dtype=torch.uint8, device=dev)
    gsx = torch.empty(1, device=dev)
    out = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    lws = torch.empty(int(B.lib().nvfp4_linear_workspace_size()), dtype=torch.uint8, device=dev)
    flush_buf = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def fn():
        B.nvfp4_quantize(x, codes=xc[:M], sf=xsf, gs_out=gsx, sf_layout=B.NVFP4_SF_TILED_ROWS)
        B.nvfp4_linear(xc, xsf, gsx, M, wc, wsf, gsw, out=out, ws=lws)
    for _ in range(args.warmup):
        fn()
    torch.cuda.synchronize()
    if B.nvfp4moe_last_device_status() != 0:
        raise RuntimeError("device status after warm-up")
    stream = torch.cuda.current_stream()
    clocks = ClockSampler(0)
    clocks.start()
    time.sleep(1.0)
    t0 = time.time()
    ms, steps = _timed(stream, args.steps, fn, flush=lambda: flush_buf.zero_(), min_seconds=1.5)
    clk = clocks.stop(t0, time.time())
    flops = 2.0 * M * N * K
    tf = flops / (ms * 1e-3) / 1e12
    peaks, kind = load_peaks()
    fp4 = float(peaks.get("bf16_tflops", 0)) * FP4_OVER_BF16
    # the GEMM alone (the dominant kernel) for the roofline
    gemm_ms, _ = _timed(stream, args.steps,
                        lambda: B.nvfp4_linear(xc, xsf, gsx, M, wc, wsf, gsw, out=out, ws=lws),
                        flush=lambda: flush_buf.zero_())
    g_tf = flops / (gemm_ms * 1e-3) / 1e12
    x_h = x.cpu().pin_memory()
    o_h = torch.empty(out.shape, dtype=torch.bfloat16).pin_memory()
    x_d = torch.empty_like(x)

    def e2e_step():
        x_d.copy_(x_h, non_blocking=True)
        B.nvfp4_quantize(x_d, codes=xc[:M], sf=xsf, gs_out=gsx, sf_layout=B.NVFP4_SF_TILED_ROWS)
        B.nvfp4_linear(xc, xsf, gsx, M, wc, wsf, gsw, out=out, ws=lws)
        o_h.copy_(out, non_blocking=True)
    e2e_step()
    e2e_ms, _ = _timed(stream, max(3, args.steps // 10), e2e_step)
    import oracle as O
    rows = 64
    xb = W.bf16_bits(x[:rows].cpu())
    c0 = time.perf_counter()
    g1 = O.global_scale(O.amax_bf16(W.bf16_bits(x.cpu())))
    wb = W.bf16_bits(inp["w"][0].cpu())
    c2, s2, g2 = O.quantize_expert(wb)
    O.matmul_nt(O.dequantize_f64(*O.quantize_bf16(xb, g1), g1), O.dequantize_f64(c2, s2, g2))
    dt = time.perf_counter() - c0
    cpu = {"value": 2.0 * rows * N * K / dt / 1e12, "unit": "TFLOP/s", "cores": O.get_threads(),
           "kind": "oracle", "sample": "%d of the %d rows (activation scale over all rows, weight "
                                       "quantization included); %.1f s" % (rows, M, dt)}
    line = _side_line(
        args, "shared-expert NVFP4 linear (quantize + GEMM) TFLOP/s", tf, "TFLOP/s", ms,
        {"workload": "linear", "M": M, "K": K, "N": N,
         "l2": "L2 flushed (256 MB written) before every timed call"},
        {"bound": "tensor", "achieved": g_tf, "peak": fp4, "unit": "TFLOP/s", "frac": g_tf / fp4,
         "traffic": None, "kernel": "grouped_gemm_kernel<false> (one group)", "kernel_ms": gemm_ms,
         "peak_source": "%s bf16 burst x 6 (nominal dense fp4/bf16 ratio)" % kind},
        {"value": flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s", "ms_per_step": e2e_ms,
         "h2d_bytes_per_step": x.numel() * 2, "d2h_bytes_per_step": out.numel() * 2},
        4 * steps, clk, cpu, steps)
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    if args.op == "qnorm_rope":
        return run_qnorm_rope(args)
    if args.op == "linear":
        return run_linear(args)
    from nvfp4_block_scaled_05_gb300 import workloads as W
    cfg = W.CONFIGS[args.workload]
    if args.impl == "reference":
        run_reference(args, cfg)
    else:
        run_ours(args, cfg)


if __name__ == "__main__":
    main()
