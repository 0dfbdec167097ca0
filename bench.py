#!/usr/bin/env python
"""Benchmark of the single-GPU MoE layer (routing -> schedule -> gather ->
grouped SwiGLU FFN -> weighted merge, forward and backward) on GB300.

Default workload: the Kimi-like layer (hidden 7168, expert intermediate 2048,
256 experts, top-8, 4,096 tokens, Zipf(1.2)-skewed routing), BF16 forward.
One step = moe_schedule + moe_forward on one batch of seeded synthetic input
already resident in HBM (fwd+bwd workloads add moe_backward).  Prints ONE
JSON line (rank 0).  `--impl reference` times the fp64 CPU oracle instead, on
a bounded sample of the same workload.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload kimi_zipf]
  python -m torch.distributed.run --nproc-per-node N bench.py --gpus N ...

Timing: W warm-up steps, then about a second of further untimed steps with
the GPU clocks sampled (so the samples see the GPU under load), then K timed
steps between CUDA events with a barrier and a synchronise on both sides and
no other work in between.  Per-kernel times come from a separate traced pass
afterwards.  With N > 1 every rank runs an independent replica of the layer
(the layer has no exchange step on one GPU); value = routed tokens of all
ranks / the slowest rank's time.
"""
import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE layer fwd/bwd ms, TFLOP/s and routed tokens/s; % of tensor peak and HBM BW"
UNIT = "routed tokens/s"

# kernel -> (flop kind, algorithmic FLOPs, algorithmic HBM bytes) per launch.
#   FLOPs: 2*M*N*K over the real (unpadded) rows.  Bytes: each weight of the
#   `touched` experts (those with rows) read once -- the weight gradients write
#   every expert's dW -- plus one read of each input row and one write of each
#   output row.  Memory-only kernels have no FLOPs.
def kernel_units(c, touched, saved=True):
    R, T, d, f, k, E = c["T"] * c["k"], c["T"], c["d"], c["f"], c["k"], c["E"]
    b = 2.0  # bf16
    w1, w2 = touched * d * 2 * f * b, touched * f * d * b
    a_out = 3 if saved else 1  # GEMM1 writes A, and H when saving
    return {
        "gemm1_swiglu": ("flop", 2.0 * R * d * 2 * f, w1 + R * d * b + R * a_out * f * b),
        "gemm2": ("flop", 2.0 * R * f * d, w2 + R * f * b + R * d * b),
        "dgrad2_dswiglu": ("flop", 2.0 * R * d * f, w2 + R * d * b + 2 * R * 3 * f * b),
        "wgrad2": ("flop", 2.0 * R * f * d, E * f * d * b + R * f * b + R * d * b),
        "wgrad1": ("flop", 2.0 * R * d * 2 * f, E * d * 2 * f * b + R * d * b + R * 2 * f * b),
        "dgrad1": ("flop", 2.0 * R * 2 * f * d, w1 + R * 2 * f * b + R * d * b),
        "gemm1_swiglu_mxfp8": ("flop8", 2.0 * R * d * 2 * f,
                               touched * d * 2 * f * (1 + 1 / 32) + R * d * (1 + 1 / 32) + R * f * (1 + 1 / 32)),
        "gemm2_mxfp8": ("flop8", 2.0 * R * f * d, touched * f * d * (1 + 1 / 32) + R * f * (1 + 1 / 32) + R * d * b),
        # gathers: one read per distinct token (its k reads after the first hit
        # L2) and one write per routed row
        "gather": (None, 0.0, T * d * b + R * d * b),
        "gather_mxfp8": (None, 0.0, T * d * b + R * d * (1.0 + 1.0 / 32)),
        "gather_x_dy": (None, 0.0, 2.0 * (T * d * b + R * d * b)),
        "merge": (None, 0.0, T * (k + 1) * d * b + R * 4.0 * 2),
        "recompute_gemm1": ("flop", 2.0 * R * d * 2 * f, w1 + R * d * b + R * 3 * f * b),
        "ring_forward_mxfp8": ("flop8", 2.0 * R * d * 2 * f + 2.0 * R * f * d,
                               T * d * b + (touched * 3 * d * f + R * f + R * d) * (1 + 1 / 32)
                               + 2.0 * R * d * b + T * d * b),
        "dgrad2_dswiglu_mxfp8": ("flop8", 2.0 * R * d * f,
                                 (touched * f * d + R * d) * (1 + 1 / 32) + R * 3 * f * b
                                 + (2 * R * 2 * f + R * f) * (1 + 1 / 32)),
        "dgrad1_mxfp8": ("flop8", 2.0 * R * 2 * f * d, (touched * d * 2 * f + R * 2 * f) * (1 + 1 / 32) + R * d * b),
        "wgrad1_mxfp8": ("flop8", 2.0 * R * d * 2 * f, E * d * 2 * f * b + (R * d + R * 2 * f) * (1 + 1 / 32)),
        "wgrad2_mxfp8": ("flop8", 2.0 * R * f * d, E * f * d * b + (R * f + R * d) * (1 + 1 / 32)),
        "quant_dy_rows": (None, 0.0, R * d * b + R * d * (1 + 1 / 32)),
        "quant_x_cols": (None, 0.0, R * d * b + R * d * (1 + 1 / 32)),
        "quant_dy_cols": (None, 0.0, R * d * b + R * d * (1 + 1 / 32)),
        "reverse_dispatch": (None, 0.0, T * (k + 1) * d * b + R * 4.0),
        # persistent ring forward (gather + GEMM1 + SwiGLU + GEMM2 + merge in one launch):
        # token rows in, weights of the touched experts, H and A saved, Y written and read
        # back by the merge, out written
        "ring_forward": ("flop", 2.0 * R * d * 2 * f + 2.0 * R * f * d,
                         T * d * b + w1 + w2 + R * a_out * f * b + 2.0 * R * d * b + T * d * b),
        # router projection (--router): x [T, d], Wr [E, d], logits / ids / weights
        "router_logits": ("flop", 2.0 * T * d * E, T * d * b + E * d * b + R * 8.0),
        "router_dlogits_bf16": (None, 0.0, T * E * 6.0),
        "router_dx": ("flop", 2.0 * T * E * d, T * E * b + E * d * b + T * d * b),
        "router_dw": ("flop", 2.0 * T * E * d, T * E * b + T * d * b + E * d * b),
    }


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            m = json.load(fh)
        return {"hbm_gbs": m["hbm_gbs"], "bf16": m["bf16_tflops"],
                "bf16_sustained": m.get("bf16_tflops_sustained", m["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16": 1900.0, "bf16_sustained": 1700.0, "source": "fallback"}


# the translation unit that defines each traced kernel
KERNEL_SOURCE = {"ring_forward": "ring.cu", "gather": "gather_merge.cu", "gather_x_dy": "gather_merge.cu",
                 "gather_mxfp8": "gather_merge.cu", "merge": "gather_merge.cu",
                 "reverse_dispatch": "gather_merge.cu", "dg_reduce": "gather_merge.cu",
                 "sched_topk_hist": "sched.cu", "sched_hist": "sched.cu", "sched_scatter": "sched.cu",
                 "sched_fused": "sched.cu",
                 "quant_dy_rows": "gather_merge.cu", "quant_x_cols": "gather_merge.cu",
                 "quant_dy_cols": "gather_merge.cu", "quantize_weights": "gather_merge.cu"}


def strip_comments(text):
    """C++ source without // and /* */ comments and blank lines (string
    literals in these sources hold no comment markers)."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(ln.rstrip() for ln in text.splitlines() if ln.strip())


def src_digest(kernel=None, read=None):
    """Digest of the code (comments stripped) a kernel is built from: its
    translation unit (gemm.cu for the grouped GEMMs) and the library headers
    it includes, directly or not; all sources when kernel is None.
    read(name) returns a source's text (default: the working tree)."""
    csrc = os.path.join(ROOT, "mixture_experts_layer_stable_gb300", "csrc")
    names = set(os.listdir(csrc))
    if read is None:
        def read(name):
            with open(os.path.join(csrc, name), encoding="utf-8") as fh:
                return fh.read()
    if kernel is None:
        files = sorted(names)
    else:
        files, todo = set(), [KERNEL_SOURCE.get(kernel, "gemm.cu")]
        while todo:
            name = todo.pop()
            if name in files or name not in names:
                continue
            files.add(name)
            todo += [os.path.basename(i) for i in re.findall(r'#include\s+"([^"]+)"', read(name))]
        files = sorted(files)
    h = hashlib.sha256()
    for name in files:
        h.update(name.encode() + strip_comments(read(name)).encode())
    return h.hexdigest()[:16]


def ncu_traffic(workload, kernel):
    """DRAM bytes per launch from a committed ncu capture, if it was taken on
    the current kernel sources (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as fh:
        tab = json.load(fh)
    ent = tab.get(f"{workload}/{kernel}")
    if not ent or ent.get("src_digest") != src_digest(kernel):
        return None
    return ent.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi samples of the SM clock and throttle reasons every 100 ms;
    stop(since) keeps the samples taken after wall time `since`."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu):
        self.gpu = gpu
        self.proc = None
        self.out = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.gpu)], stdout=self.out, stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None

    @staticmethod
    def parse(lines, since=None):
        """Summary of sample lines (timestamp first; local time as nvidia-smi
        prints it); samples before wall time `since` are dropped."""
        sm, mx, pw, reasons = [], 0.0, [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in lines:
            r = [c.strip() for c in line.split(",")]
            try:
                ts = time.mktime(time.strptime(r[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                ts += float("0." + r[0].split(".")[1]) if "." in r[0] else 0.0
                if since is not None and ts < since:
                    continue
                sm.append(float(r[2]))
                mx = max(mx, float(r[3]))
                pw.append(float(r[4]))
                for nm, v in zip(names, r[6:10]):
                    if v.lower() == "active":
                        reasons.add(nm)
            except (ValueError, IndexError):
                continue
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "sm_mhz_min": min(sm),
                "power_w_median": statistics.median(pw), "reasons": sorted(reasons),
                "samples": len(sm)}

    def stop(self, since=None):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.flush()
        self.out.seek(0)
        lines = [l for l in self.out.read().splitlines() if l.strip()]
        os.unlink(self.out.name)
        return self.parse(lines, since)


def workload_dict(cfg):
    return {"T": cfg.T, "d": cfg.d, "f": cfg.f, "E": cfg.E, "k": cfg.k}


# --------------------------------------------------------------- the oracle
def oracle_sample(cfg, n_experts, seed=0):
    """CPU inputs of the workload for the first n_experts experts (the same
    seeded draws as the full workload) -- used only by the CPU baseline."""
    import torch
    from mixture_experts_layer_stable_gb300.inputs import make_inputs
    inp = make_inputs(cfg, device="cpu", seed=seed, parts=("logits", "x", "dOut"))
    w = make_inputs(cfg, device="cpu", seed=seed, parts=("W1", "W2"), experts=n_experts)
    inp.update(w)
    return inp


def oracle_step(cfg, inp, experts, passes="fwd+bwd"):
    """One oracle pass over a sample: routing + schedule for every token,
    then the forward (and, for fwd+bwd, the backward) of every row routed to
    `experts`.  Returns the number of routed rows processed."""
    import torch
    from oracle import moe_oracle as O

    ids, g = O.route(inp["logits"].numpy(), cfg.k)
    counts, offsets, perm, inv = O.schedule(ids, cfg.E)
    x = inp["x"].to(torch.float64).numpy()
    W1 = lambda e: inp["W1"][e].to(torch.float64).numpy()
    W2 = lambda e: inp["W2"][e].to(torch.float64).numpy()
    if passes == "fwd":
        for e in experts:
            a, b = int(offsets[e]), int(offsets[e + 1])
            if a < b:
                O.expert_ffn(x[perm[a:b] // cfg.k], W1(e), W2(e))
    else:
        class View:
            def __len__(self):
                return cfg.E

            def __getitem__(self, e):
                return W1(e) if self.which == 1 else W2(e)

        v1, v2 = View(), View()
        v1.which, v2.which = 1, 2
        dO = inp["dOut"].to(torch.float64).numpy()
        O.backward_experts(x, v1, v2, ids, g, dO, list(experts))
    return int(sum(int(counts[e]) for e in experts))


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count()


def time_oracle(cfg, budget_s, steps=1, warmup=0, passes="fwd+bwd"):
    """Pick the sample -- the rows of experts 0..n-1 -- so that one oracle
    pass takes about budget_s, run warmup + steps passes, return (rows/s,
    sample description, seconds)."""
    import numpy as np
    from oracle import moe_oracle as O
    inp = oracle_sample(cfg, 1)
    ids, _ = O.route(inp["logits"].numpy(), cfg.k)
    counts = np.bincount(ids.reshape(-1), minlength=cfg.E)
    # cost of one row: from the first nonempty expert's rows (at most 256 of them)
    e0 = int(np.argmax(counts > 0))
    inp = oracle_sample(cfg, e0 + 1)
    oracle_step(cfg, inp, [e0], passes)             # first call: BLAS start-up
    t0 = time.perf_counter()
    rows1 = oracle_step(cfg, inp, [e0], passes)
    per_row = max(time.perf_counter() - t0, 1e-4) / max(rows1, 1)
    n = 1
    while n < cfg.E and (np.cumsum(counts)[n] * per_row) <= budget_s:
        n += 1
    inp = oracle_sample(cfg, n)
    experts = range(n)
    for _ in range(warmup):
        oracle_step(cfg, inp, experts, passes)
    rows = 0
    t0 = time.perf_counter()
    for _ in range(steps):
        rows += oracle_step(cfg, inp, experts, passes)
    dt = time.perf_counter() - t0
    what = "forward" if passes == "fwd" else "forward+backward"
    desc = (f"routing + schedule of all {cfg.T} tokens, then {what} (fp64 numpy) of the rows "
            f"routed to experts 0..{n - 1} of {cfg.E}; {rows // max(steps, 1)} of {cfg.T * cfg.k} "
            f"routed rows per pass")
    return rows / dt, desc, dt


# --------------------------------------------------------------- main
def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="kimi_zipf")
    ap.add_argument("--passes", default=None, help="fwd or fwd+bwd (default: the workload's)")
    ap.add_argument("--prec", choices=["bf16", "mxfp8"], default=None,
                    help="precision (default: the workload's)")
    ap.add_argument("--save", action="store_true",
                    help="forward-only passes: also save H and A for a later backward")
    ap.add_argument("--minibatch-rows", type=int, default=0,
                    help="0 = the kernel chain; > 0 = the forward through the persistent ring "
                         "kernel with windows of this many expert-ordered rows")
    ap.add_argument("--ring-slots", type=int, default=4)
    ap.add_argument("--gather-ctas", type=int, default=0, help="ring: 0 = gather warps in every CTA, G > 0 = G gather-only CTAs")
    ap.add_argument("--settle-s", type=float, default=1.0,
                    help="seconds of untimed steps after the warm-up, clocks sampled")
    ap.add_argument("--tile-scheduler", choices=["static", "clc"], default=None,
                    help="how the one-CTA weight-gradient GEMMs take their tiles (default: the library's)")
    ap.add_argument("--no-graph", action="store_true",
                    help="launch every step's calls eagerly instead of replaying them as one CUDA graph")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--router", action="store_true",
                    help="route from x and a router weight (moe_route, plus the router backward) "
                         "instead of from the workload's synthetic logits")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=None)
    return ap.parse_args()


def max_over_ranks(x, dist=None, device="cpu"):
    """The largest x over all ranks (x itself without a process group)."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(rows_per_step, steps, world, ms_max):
    """Whole-job routed rows/s: every rank's rows over the slowest rank's time."""
    return rows_per_step * steps * world / (ms_max / 1000.0)


def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def run_reference(args, cfg, rank):
    if rank != 0:
        return
    passes = args.passes or cfg.passes
    budget = 0.5 if args.steps + args.warmup <= 200 else max(0.05, 100.0 / (args.steps + args.warmup))
    v, desc, dt = time_oracle(cfg, budget, steps=args.steps, warmup=args.warmup, passes=passes)
    cores = blas_threads()
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 * dt / max(args.steps, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded torch generators; no dataset)",
        "config": {"workload": cfg.name, **workload_dict(cfg), "passes": passes},
        "cpu_baseline": {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc},
        "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    world, rank, local = dist_setup()
    from mixture_experts_layer_stable_gb300.configs import CONFIGS
    cfg = CONFIGS[args.workload]
    if args.prec and args.prec != cfg.prec:
        import dataclasses
        cfg = dataclasses.replace(cfg, prec=args.prec)
    passes = args.passes or cfg.passes
    if args.impl == "reference":
        run_reference(args, cfg, rank)
        return

    import torch
    import __graft_entry__
    __graft_entry__.build()
    from mixture_experts_layer_stable_gb300 import binding as B
    from mixture_experts_layer_stable_gb300.inputs import make_inputs

    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    if args.tile_scheduler is not None:
        B.moe_set_tile_scheduler(1 if args.tile_scheduler == "clc" else 0)
    prec = B.MOE_MXFP8 if cfg.prec == "mxfp8" else B.MOE_BF16
    bwd = passes != "fwd"
    save = bwd or args.save
    mb = args.minibatch_rows
    c = B.make_config(cfg.T, cfg.d, cfg.f, cfg.E, cfg.k, prec, mb,
                      args.ring_slots if mb > 0 else 0, args.gather_ctas)
    inp = make_inputs(cfg, device="cuda", seed=0, with_grad=bwd)
    w1, w1s, w2, w2s = inp["W1"], None, inp["W2"], None
    if cfg.prec == "mxfp8":
        # weights pre-quantised once along K (E4M3 + UE8M0 per 32), outside the timed region
        w1 = torch.empty(cfg.E, 2 * cfg.f, cfg.d, dtype=torch.uint8, device="cuda")
        w1s = torch.empty(cfg.E * 2 * cfg.f * cfg.d // 32, dtype=torch.uint8, device="cuda")
        w2 = torch.empty(cfg.E, cfg.d, cfg.f, dtype=torch.uint8, device="cuda")
        w2s = torch.empty(cfg.E * cfg.d * cfg.f // 32, dtype=torch.uint8, device="cuda")
        B.moe_quantize_mxfp8(inp["W1"], cfg.E, cfg.d, 2 * cfg.f, w1, w1s)
        B.moe_quantize_mxfp8(inp["W2"], cfg.E, cfg.f, cfg.d, w2, w2s)
        if bwd:
            # the backward's copies, quantised along the other dimension
            w1r = torch.empty(cfg.E, cfg.d, 2 * cfg.f, dtype=torch.uint8, device="cuda")
            w1rs = torch.empty(cfg.E * cfg.d * 2 * cfg.f // 32, dtype=torch.uint8, device="cuda")
            w2r = torch.empty(cfg.E, cfg.f, cfg.d, dtype=torch.uint8, device="cuda")
            w2rs = torch.empty(cfg.E * cfg.f * cfg.d // 32, dtype=torch.uint8, device="cuda")
            B.moe_quantize_mxfp8_rows(inp["W1"], cfg.E * cfg.d, 2 * cfg.f, w1r, w1rs)
            B.moe_quantize_mxfp8_rows(inp["W2"], cfg.E * cfg.f, cfg.d, w2r, w2rs)
    sched = B.alloc_sched(c)
    ws = B.alloc_workspace(c)
    saved = B.alloc_saved(c) if save else None
    out = torch.empty(cfg.T, cfg.d, dtype=torch.bfloat16, device="cuda")
    if bwd:
        dx = torch.empty_like(out)
        dW1 = torch.empty_like(inp["W1"])
        dW2 = torch.empty_like(inp["W2"])
        dtw = torch.empty(cfg.T * cfg.k, dtype=torch.float32, device="cuda")
        dlog = torch.empty(cfg.T, cfg.E, dtype=torch.float32, device="cuda")

    if args.router:
        gr = torch.Generator(device="cuda").manual_seed(5)
        w_router = (torch.randn(cfg.E, cfg.d, device="cuda", generator=gr) / cfg.d ** 0.5).to(torch.bfloat16)
        r_logits = None if cfg.E <= 256 else torch.empty(cfg.T, cfg.E, dtype=torch.float32, device="cuda")
        if bwd:
            dx_r = torch.empty(cfg.T, cfg.d, dtype=torch.bfloat16, device="cuda")
            dw_r = torch.empty_like(w_router)

    def step(logits=inp["logits"], x=inp["x"], dOut=inp.get("dOut"), out_=None, dx_=None):
        o = out if out_ is None else out_
        if args.router:
            B.moe_route(c, x, w_router, r_logits, sched, ws)
        else:
            B.moe_schedule(c, logits, sched, ws)
        B.moe_forward(c, x, w1, w1s, w2, w2s, sched, o, saved, ws)
        if bwd:
            g = dx if dx_ is None else dx_
        if bwd and cfg.prec == "mxfp8":
            B.moe_backward_mxfp8(c, dOut, x, w1r, w1rs, w2r, w2rs, sched, saved, g, dW1, dW2, dtw, dlog, ws)
        elif bwd:
            B.moe_backward(c, dOut, x, w1, w2, sched, saved, g, dW1, dW2, dtw, dlog, ws)
            if args.router:
                B.moe_router_backward(c, x, w_router, dlog, dx_r, dw_r, ws)

    # ---------------- the step as one CUDA graph: the library's calls are
    # capturable (no synchronisation, no allocation); replaying the graph
    # removes the host's per-call launch work from the step
    graph = None
    graph_note = "eager launches"
    if not args.no_graph:
        step()  # first calls outside capture: kernel attributes, occupancy queries
        torch.cuda.synchronize()
        try:
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                step()
            graph_note = "one CUDA graph per step (captured library calls)"
        except Exception as ex:  # pragma: no cover - depends on the CUDA version
            graph = None
            graph_note = f"eager launches (graph capture failed: {type(ex).__name__})"
            torch.cuda.synchronize()

    def run_step():
        if graph is not None:
            graph.replay()
        else:
            step()

    # ---------------- warm-up, then untimed steps with the clocks sampled
    wa, wb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for i in range(max(args.warmup, 1)):
        run_step()
        if i == 0:
            wa.record()
    wb.record()
    torch.cuda.synchronize()
    st = B.moe_read_status(ws)
    if st != 0:
        raise RuntimeError(f"device status after warm-up: {B.moe_status_string(st)}")
    est_ms = wa.elapsed_time(wb) / max(args.warmup - 1, 1) if args.warmup > 1 else 5.0
    gpu_idx = local
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        try:
            gpu_idx = int(vis.split(",")[local])
        except ValueError:
            pass
    clocks = ClockSampler(gpu_idx)
    clocks.start()
    time.sleep(0.2)  # the sampler's first line comes after nvidia-smi starts up
    t_load = time.time()
    n_settle = int(min(20000, max(0, args.settle_s * 1000.0 / max(est_ms, 1e-3))))
    for _ in range(n_settle):
        run_step()

    # ---------------- timed region (device-resident inputs, no tracing)
    barrier()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record()
    for _ in range(args.steps):
        run_step()
    ev1.record()
    barrier()
    clk = clocks.stop(since=t_load)
    if clk is not None:
        clk["window"] = "%d untimed steps (%.2f s) + the timed region" % (n_settle, n_settle * est_ms / 1e3)
    ms = ev0.elapsed_time(ev1)
    st = B.moe_read_status(ws)
    if st != 0:
        raise RuntimeError(f"device status after timed region: {B.moe_status_string(st)}")
    ms_max = max_over_ranks(ms, dist, "cuda")
    R = cfg.T * cfg.k
    value = job_throughput(R, args.steps, world, ms_max)
    ms_step = ms_max / args.steps

    # ---------------- per-kernel times: a separate traced pass
    n_tr = max(3, min(args.steps, 20))
    B.moe_trace_enable(0)
    B.moe_trace_enable(64 * n_tr + 64)
    for _ in range(n_tr):
        step()
    torch.cuda.synchronize()
    n_launch = B.moe_trace_count()
    per = {}
    for i in range(n_launch):
        name, kms = B.moe_trace_read(i)
        a = per.setdefault(name, [0, 0.0])
        a[0] += 1
        a[1] += kms
    B.moe_trace_enable(0)
    launches_per_step = n_launch / n_tr

    # ---------------- end to end through the C ABI with host buffers
    # Every step copies its inputs (logits, x; dOut with the backward) from
    # pinned host memory and its results (out; dx) back.  Two buffer sets
    # alternate, so that a step's host-to-device copies (one copy stream)
    # overlap the previous step's kernels and its device-to-host copies (a
    # second copy stream) the next step's, as a pipeline feeding the layer
    # would run; each step's own copies stay inside the timed region.
    e2e = None
    if not args.no_e2e:
        names = ("logits", "x", "dOut") if bwd else ("logits", "x")
        k_e2e = args.e2e_steps or max(10, args.steps // 4)
        host_in = [{k: inp[k].cpu().pin_memory() for k in names} for _ in range(2)]
        dev_in = [{k: inp[k] for k in names}, {k: torch.empty_like(inp[k]) for k in names}]
        dev_out = [out, torch.empty_like(out)]
        dev_dx = [dx, torch.empty_like(dx)] if bwd else [None, None]
        host_out = [torch.empty(out.shape, dtype=out.dtype, pin_memory=True) for _ in range(2)]
        host_dx = ([torch.empty(out.shape, dtype=out.dtype, pin_memory=True) for _ in range(2)]
                   if bwd else [None, None])
        h2d = sum(t.numel() * t.element_size() for t in host_in[0].values())
        d2h = host_out[0].numel() * 2 + (host_dx[0].numel() * 2 if bwd else 0)
        graphs = [graph, None]
        if graph is not None:
            g1 = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g1):
                step(dev_in[1]["logits"], dev_in[1]["x"], dev_in[1].get("dOut"), dev_out[1], dev_dx[1])
            graphs[1] = g1
        comp = torch.cuda.current_stream()
        up, down = torch.cuda.Stream(), torch.cuda.Stream()
        ev_in = [torch.cuda.Event() for _ in range(2)]
        ev_done = [torch.cuda.Event() for _ in range(2)]
        ev_out = [torch.cuda.Event() for _ in range(2)]

        def e2e_step(i):
            b = i & 1
            with torch.cuda.stream(up):
                up.wait_event(ev_done[b])  # the step that last read set b is done
                for k_, t in host_in[b].items():
                    dev_in[b][k_].copy_(t, non_blocking=True)
                ev_in[b].record(up)
            comp.wait_event(ev_in[b])
            comp.wait_event(ev_out[b])  # set b's previous results have left
            if graphs[b] is not None:
                graphs[b].replay()
            else:
                step(dev_in[b]["logits"], dev_in[b]["x"], dev_in[b].get("dOut"), dev_out[b], dev_dx[b])
            ev_done[b].record(comp)
            with torch.cuda.stream(down):
                down.wait_event(ev_done[b])
                host_out[b].copy_(dev_out[b], non_blocking=True)
                if bwd:
                    host_dx[b].copy_(dev_dx[b], non_blocking=True)
                ev_out[b].record(down)

        for i in range(3):
            e2e_step(i)
        torch.cuda.synchronize()
        barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(comp)
        up.wait_stream(comp)  # the first copies start after the timer
        for i in range(k_e2e):
            e2e_step(i)
        comp.wait_event(ev_out[0])
        comp.wait_event(ev_out[1])
        e1.record(comp)
        torch.cuda.synchronize()
        barrier()
        ems = max_over_ranks(e0.elapsed_time(e1), dist, "cuda")
        e2e = {"value": job_throughput(R, k_e2e, world, ems), "unit": UNIT,
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "steps": k_e2e,
               "copies": "pinned host buffers, two sets alternating; a step's H2D and D2H copies "
                         "run on two copy streams beside the neighbouring steps' kernels"}

    # ---------------- per-kernel roofline
    # the binding resource of each kernel is the larger of FLOPs / tensor peak
    # and algorithmic bytes / HBM bandwidth; kernels run inside a long loop of
    # steps, so the tensor peak is the sustained one
    peaks = load_peaks()
    touched = int((sched["counts"] > 0).sum().item())
    units = kernel_units(workload_dict(cfg), touched, saved=save)

    def roof_of(name, avg_ms):
        kind, flop, nbytes = units[name]
        fpeak = peaks["bf16_sustained"] * (2.0 if kind == "flop8" else 1.0)
        t_f = flop / (fpeak * 1e12) if kind else 0.0
        t_b = nbytes / (peaks["hbm_gbs"] * 1e9)
        tr = ncu_traffic(cfg.name, name)
        dram = None if tr is None else tr / (avg_ms / 1e3) / 1e9 / peaks["hbm_gbs"]
        if t_f >= t_b:
            src = (f"{peaks['source']} bf16 sustained (MEASURED_PEAKS.json)" if kind == "flop" else
                   f"{peaks['source']} bf16 sustained x 2 (nominal fp8:bf16 dense ratio 4.5:2.25)")
            ach = flop / (avg_ms / 1e3) / 1e12
            return {"bound": "tensor", "achieved": ach, "peak": fpeak, "unit": "TFLOP/s",
                    "frac": ach / fpeak, "algorithmic_per_launch": flop, "peak_source": src,
                    "hbm_frac": nbytes / (avg_ms / 1e3) / 1e9 / peaks["hbm_gbs"],
                    "dram_frac_ncu": dram}
        ach = nbytes / (avg_ms / 1e3) / 1e9
        return {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": ach / peaks["hbm_gbs"], "algorithmic_per_launch": nbytes,
                "peak_source": f"{peaks['source']} hbm copy (MEASURED_PEAKS.json)",
                "tensor_frac": (flop / (avg_ms / 1e3) / 1e12 / fpeak) if kind else None,
                "dram_frac_ncu": dram}

    kernels = {}
    tot_all = max(sum(v[1] for v in per.values()), 1e-9)
    for name, (cnt, tot) in per.items():
        avg = tot / cnt
        ent = {"launches": cnt, "ms_per_launch": avg, "share": tot / tot_all}
        if name in units:
            r = roof_of(name, avg)
            ent.update({"bound": r["bound"], "frac": r["frac"], r["unit"]: r["achieved"]})
            if r.get("dram_frac_ncu") is not None:
                ent["dram_frac_ncu"] = r["dram_frac_ncu"]
        kernels[name] = ent
    dom = max(per.items(), key=lambda kv: kv[1][1])[0]
    avg = per[dom][1] / per[dom][0]
    roof = roof_of(dom, avg) if dom in units else {"bound": None, "frac": None}
    tr = ncu_traffic(cfg.name, dom)
    roof.update({"traffic": tr, "kernel": dom,
                 "timing": "CUDA events around each launch on its stream, traced pass of %d steps "
                           "after the timed region" % n_tr})
    fwd_names = ("gather", "gather_mxfp8", "gemm1_swiglu", "gemm2", "gemm1_swiglu_mxfp8",
                 "gemm2_mxfp8", "merge", "ring_forward", "ring_forward_mxfp8")
    sched_names = ("sched_fused", "sched_topk_hist", "sched_hist", "sched_scatter", "router_logits")
    fwd_ms = sum(per[n][1] for n in per if n in fwd_names) / n_tr
    sch_ms = sum(per[n][1] for n in per if n in sched_names) / n_tr
    bwd_ms = sum(per[n][1] for n in per if n not in fwd_names + sched_names) / n_tr
    flops = (6.0 if not bwd else 18.0) * R * cfg.d * cfg.f
    if args.router:
        flops += (2.0 if not bwd else 6.0) * cfg.T * cfg.d * cfg.E
    tflops = flops / (ms_step / 1e3) / 1e12
    fpk = 2.0 if cfg.prec == "mxfp8" else 1.0
    # the layer's own bound: its FLOPs at the tensor peak against streaming
    # the touched experts' weights once (bf16: 6 d f bytes each; mxfp8: 3 d f
    # plus scales) at the HBM bandwidth
    wbytes = touched * 3.0 * cfg.d * cfg.f * (2.0 if cfg.prec == "bf16" else (1 + 1 / 32))
    if bwd:
        wbytes += cfg.E * 6.0 * cfg.d * cfg.f  # every dW written once
    layer = {"tflops": tflops,
             "tensor_frac_sustained": tflops / (peaks["bf16_sustained"] * fpk),
             "tensor_frac_burst": tflops / (peaks["bf16"] * fpk),
             "peak_note": ("MXFP8 against 2x the bf16 peaks (nominal fp8:bf16 dense ratio 4.5:2.25)"
                          if cfg.prec == "mxfp8" else "bf16 peaks of MEASURED_PEAKS.json"),
             "weight_stream_ms": wbytes / (peaks["hbm_gbs"] * 1e9) * 1e3,
             "flop_ms_burst": flops / (peaks["bf16"] * fpk * 1e12) * 1e3,
             "experts_touched": touched}

    # ---------------- CPU baseline: the oracle on a bounded sample
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, desc, dt = time_oracle(cfg, 12.0, steps=1, passes=passes)
        cpu = {"value": v, "unit": UNIT, "cores": blas_threads(), "kind": "oracle", "sample": desc,
               "seconds": dt}

    if rank != 0:
        return
    fwd_desc = ("persistent ring kernel, %d-row windows, %d slots, %s" % (
        mb, args.ring_slots, "%d gather CTAs" % args.gather_ctas if args.gather_ctas > 0
        else "gather warps in every CTA") if mb > 0 else "kernel chain")
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "e4m3 (mxfp8)" if cfg.prec == "mxfp8" else "bf16",
        "data": "synthetic (seeded torch generators on device; no dataset, random-init weights)",
        "config": {"workload": cfg.name, **workload_dict(cfg), "passes": passes, "prec": cfg.prec,
                   "minibatch_rows": mb, "forward": fwd_desc, "launch": graph_note,
                   "tile_scheduler": ["static walk", "cluster launch control"][B.moe_get_tile_scheduler()],
                   "saved_activations": "H and A" if save else "none",
                   "routing": "router projection (moe_route)" if args.router else "synthetic logits",
                   "l2": "inputs larger than L2 (weights %.2f GB per step)" % (
                       (inp["W1"].numel() + inp["W2"].numel()) * 2 / 1e9),
                   "parallelism": f"replicas x{world}"},
        "tflops": tflops, "layer": layer,
        "sched_ms": sch_ms, "fwd_ms": fwd_ms, "bwd_ms": bwd_ms,
        "roofline": roof, "kernels": kernels,
        "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": int(round(launches_per_step * args.steps)), "clocks": clk,
    }
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
