"""Benchmark of the MoE layer hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--path fused|unfused] [--cpu-sample-tokens N]
                    [--no-cpu-baseline]

One step = one full forward + backward of the layer (router, top-k gating,
permutation, grouped SwiGLU experts + shared expert, combine, and every
backward step) over one batch of seeded synthetic input, through the C ABI.
Default workload: the largest layer of the workload table, forward +
backward (T=8192, d=4096, E=128, top-4, H=Hs=1536, learned router).  Inputs
are resident in HBM when the timed region starts; L2 (129 MB) is flushed by
writing a 256 MB buffer before every step.

Two call sequences compute the same step (identical results): "fused", the
permutation inside the GEMMs' operand loads (TMA row gathers from x and dY)
and the combine inside the shared expert's down-projection epilogue
(moe_grouped_swiglu_fused, the gather mode of moe_grouped_swiglu_bwd), and
"unfused", with x_perm / dY_perm / o_perm / s written and read back
(moe_permute rows, moe_grouped_swiglu, moe_unpermute_combine and
moe_unpermute_combine_bwd).  --path picks the one the line reports (default
unfused, the faster on GB300: the row gathers cannot feed the tensor cores
at the rate of tiled TMA loads); the other is timed too (`other_path`).

`value` times the step's calls captured once in a CUDA graph and replayed
(the calls are asynchronous and allocate nothing); `fwd_tokens_per_s` does
the same for the forward calls alone.  `kernels` times every kernel launch
of the step with CUDA events that the library records just before each of
its launches (moe_timing_begin), captured as event-record nodes in a graph
of the step and replayed like the timed region; `roofline` is the kernel
with the largest share of the step, against the binding roof (tensor or HBM)
of its algorithmic work, with the measured burst peaks.

Prints ONE JSON line (rank 0).  With --gpus N > 1 (torchrun) every rank runs an
independent replica of the layer on its own tokens (weak scaling; the layer
has no exchange step, so no collective runs on the data path).

--impl reference times the CPU oracle (the C++ fp64 layer of
oracle/moe_oracle.cpp on all host cores) on a bounded token sample of the same
workload: rank 0 only.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from synth import workloads  # noqa: E402

METRIC = "MoE layer tokens/s fwd & fwd+bwd on 1 GB300; grouped-GEMM % BF16 peak"
L2_FLUSH_BYTES = 256 << 20
REFERENCE_BUDGET_S = 150.0  # CPU seconds the whole --impl reference run aims at


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="large_E128", choices=sorted(workloads.WORKLOADS))
    ap.add_argument("--cpu-sample-tokens", type=int, default=0,
                    help="oracle tokens per step (0: sized for ~20 s of CPU work)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--path", default="unfused", choices=["fused", "unfused"])
    ap.add_argument("--no-other-path", action="store_true", help="do not time the other call sequence")
    return ap.parse_args()


def backward_workload(name):
    base = workloads.WORKLOADS[name]
    return workloads.custom(base.name, T=base.T, d=base.d, E=base.E, k=base.k, H=base.H, Hs=base.Hs,
                            routing=base.routing, zipf_bias=base.zipf_bias, capacity_factor=base.capacity_factor,
                            backward=True)


# ------------------------------------------------------------------ accounting
def gemm_flops(w, R):
    """Algorithmic tensor-core FLOPs of one forward and one backward pass."""
    fwd = 6.0 * R * w.d * w.H + 6.0 * w.T * w.d * w.Hs
    bwd = 12.0 * R * w.d * w.H + 12.0 * w.T * w.d * w.Hs
    if w.routing == "learned":
        fwd += 2.0 * w.T * w.d * w.E
        bwd += 4.0 * w.T * w.d * w.E
    return fwd, bwd


def kernel_work(w, R, fused=False):
    """Algorithmic work of one launch of each kernel of the step: (FLOPs,
    bytes).  FLOPs count the method's products once (the second MMA of a
    hi + lo split operand is not counted).  Bytes count every operand read
    once and every output written once, with activations in bf16 (the
    method's own dtype) and weights and weight gradients in bf16."""
    T, d, E, k, H, Hs = w.T, w.d, w.E, w.k, w.H, w.Hs
    sh = 1 if Hs else 0
    rows = R + T * sh                                # routed rows + shared-expert rows
    wgu = 2 * (E * H * d + Hs * d) * 2               # W_g and W_u (routed + shared)
    wdn = (E * H * d + Hs * d) * 2                   # W_d
    gu = 4.0 * d * (R * H + T * Hs)
    dn = 2.0 * d * (R * H + T * Hs)
    hid = R * H + T * Hs                             # hidden elements (routed + shared)
    # the weight gradients' token operand: x_perm / dY_perm rows, or (fused)
    # the gathered source read once
    tok = T * d * 2 * (1 + sh) if fused else rows * d * 2
    return {
        "gemm_gate_up_swiglu": (gu, R * d * 2 + T * d * 2 * sh + wgu + hid * 2 + 2 * hid * 2),
        "gemm_gate_up_recompute": (gu, R * d * 2 + T * d * 2 * sh + wgu + 2 * hid * 2),
        "gemm_down": (dn, hid * 2 + wdn + rows * d * 2),
        "gemm_dgrad_down_swiglu_bwd": (dn, rows * d * 2 + wdn + 2 * hid * 2 + 2 * hid * 2 + hid * 2),
        "gemm_wgrad_down": (dn, tok + hid * 2 + wdn),
        "gemm_dgrad_gate_up": (gu, 2 * hid * 2 + wgu + rows * d * 2),
        "gemm_wgrad_gate_up": (gu, 2 * hid * 2 + tok + wgu),
        "gemm_router": (2.0 * T * d * E, T * d * 2 + E * d * 2 + T * E * 4),
        "gemm_router_dw": (2.0 * T * d * E, T * E * 2 + T * d * 2 + E * d * 4),
        "gemm_router_dx": (2.0 * T * d * E, T * E * 4 + E * d * 2 + T * d * 2),
        "perm_scatter": (0.0, T * d * 2 + R * d * 2 + T * k * 12 + R * 4),
        "combine": (0.0, R * d * 2 + T * d * 2 * sh + T * d * 2 + T * k * 8),
        "gather_rows": (0.0, T * d * 2 + R * d * 2 + T * k * 4),
        "unpermute_reduce": (0.0, R * d * 2 + T * d * 2 * sh + T * d * 2 + T * k * 4),
        "topk_gating": (0.0, T * E * 4 + T * k * 8),
        "grad_amax": (0.0, T * d * 2),  # the scale word of the backward's fp16 terms: dY read once
        # MXFP8 forward: E4M3 operands (1 byte) with one scale byte per 32
        "gemm_mx_gate_up_swiglu": (gu, (R * d + T * d * sh) * 33 // 32 + wgu // 2 * 33 // 32
                                   + hid * 33 // 32),
        "gemm_mx_down": (dn, hid * 33 // 32 + wdn // 2 * 33 // 32 + rows * d * 2),
        "perm_scatter_mx": (0.0, T * d * 2 + R * d * 33 // 32 + T * k * 12 + R * 4),
        # fused path: a gathered operand's algorithmic bytes are its source
        # (x or dY, T rows) read once; the expert outputs by slot
        "perm_maps": (0.0, T * k * 12 + R * 4),
        "gemm_gate_up_swiglu_gather": (gu, T * d * 2 * (1 + sh) + wgu + hid * 2 + 2 * hid * 2),
        "gemm_gate_up_recompute_gather": (gu, T * d * 2 * (1 + sh) + wgu + 2 * hid * 2),
        "gemm_down_slots": (2.0 * d * R * H, R * H * 2 + E * H * d * 2 + R * d * 2),
        "gemm_down_shared_combine": (2.0 * d * T * Hs, T * Hs * 2 + Hs * d * 2 + R * d * 2 + T * d * 2 + T * k * 8),
        "combine_slots": (0.0, R * d * 2 + T * d * 2 + T * k * 8),
        "gemm_dgrad_down_swiglu_bwd_gather": (dn, T * d * 2 * (1 + sh) + wdn + 2 * hid * 2 + 2 * hid * 2 + hid * 2),
    }


def issued_mma_flops(w, R):
    """MMA FLOPs the split-precision kernels issue per launch, where that is
    more than their algorithmic FLOPs: every K step of a bf16 hi + lo operand
    is issued twice (weight gradients: all tiles; dgrad of gate/up: the shared
    expert's tiles; router weight gradient and router dx: dlogits).  Tile
    padding is not counted."""
    T, d, E, k, H, Hs = w.T, w.d, w.E, w.k, w.H, w.Hs
    gu = 4.0 * d * (R * H + T * Hs)
    dn = 2.0 * d * (R * H + T * Hs)
    out = {
        "gemm_wgrad_gate_up": 2 * gu,
        "gemm_wgrad_down": 2 * dn,
        "gemm_dgrad_gate_up": 4.0 * d * (R * H + 2 * T * Hs),
        "gemm_router_dw": 2 * 2.0 * T * d * E,
        "gemm_router_dx": 2 * 2.0 * T * d * E,
    }
    out["gemm_wgrad_gate_up (gather)"] = out["gemm_wgrad_gate_up"]
    out["gemm_wgrad_down (gather)"] = out["gemm_wgrad_down"]
    return out


def with_issued(row, name, issued, ms, tensor_peak):
    """Adds the issued MMA FLOPs of a split-precision kernel and their
    fraction of the tensor peak (beside the algorithmic fraction)."""
    if name in issued:
        row["issued_mma_flops"] = issued[name]
        row["issued_tensor_frac"] = round(issued[name] / (ms / 1000.0) / (tensor_peak * 1e12), 4)
    return row


def kernel_roofline(work, ms, tensor_peak, hbm_peak):
    """Binding roof of one launch: its algorithmic FLOPs at the tensor peak
    against its algorithmic bytes at the HBM peak; `frac` = the binding roof's
    time over the measured time (= achieved / peak on that roof)."""
    flops, nbytes = work
    s = ms / 1000.0
    t_tensor = flops / (tensor_peak * 1e12)
    t_hbm = nbytes / (hbm_peak * 1e9)
    if t_tensor >= t_hbm:
        return {"bound": "tensor", "achieved": round(flops / s / 1e12, 1), "peak": tensor_peak, "unit": "TFLOP/s",
                "frac": round(t_tensor / s, 4), "hbm_frac": round(t_hbm / s, 4),
                "algorithmic_flops": flops, "algorithmic_bytes": nbytes}
    return {"bound": "hbm", "achieved": round(nbytes / s / 1e9, 1), "peak": hbm_peak, "unit": "GB/s",
            "frac": round(t_hbm / s, 4), "tensor_frac": round(t_tensor / s, 4),
            "algorithmic_flops": flops, "algorithmic_bytes": nbytes}


def profiled_traffic(workload_name, kernel):
    """DRAM bytes per launch of `kernel` on this workload from the committed ncu
    summaries under profiles/ (lines `traffic <kernel> <workload> <bytes per
    launch> <source fingerprint>`), or None when no summary covers it or the
    sources that kernel compiles from have changed since it was taken."""
    import glob
    from top_routing_grouped_moe_gb300 import build
    fp = build.kernel_fingerprint(kernel)
    for path in sorted(glob.glob(os.path.join(ROOT, "profiles", "*.md"))):
        for line in open(path):
            parts = line.split()
            if (len(parts) == 5 and parts[0] == "traffic" and parts[1] == kernel and parts[2] == workload_name
                    and parts[4] == fp):
                return int(parts[3])
    return None


# ------------------------------------------------------------------ ranks
def max_over_ranks(values, device):
    """Element-wise max of a list of floats over all ranks (identity with one
    rank).  The timed region of every rank is compared, the slowest counts."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def tokens_per_s(T, steps, world, total_ms):
    """Whole-job throughput: every rank processes T tokens per step."""
    return T * steps * world / (total_ms / 1000.0)


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu_index = gpu_index
        self.proc = None
        # the raw samples go to MOE_BENCH_CLOCKS_CSV (kept) or a temporary
        # file (removed once summarised)
        self.keep = os.environ.get("MOE_BENCH_CLOCKS_CSV")
        if self.keep:
            self.path = self.keep.replace("{rank}", str(gpu_index))
        else:
            fd, self.path = tempfile.mkstemp(prefix=f"moe_clocks_{gpu_index}_", suffix=".csv")
            os.close(fd)

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader",
                 "-lms", "50"], stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def _discard(self):
        if not self.keep:
            try:
                os.remove(self.path)
            except OSError:
                pass

    def stop(self):
        if self.proc is None:
            self._discard()
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, smax, power, reasons = [], [], [], set()
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1].split()[0]))
                smax.append(float(parts[2].split()[0]))
                power.append(float(parts[3].split()[0]))
            except ValueError:
                continue
            for name, v in zip(("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"),
                               parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        self._discard()
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": max(power) if power else None}


# ------------------------------------------------------------------ reference arm (the oracle)
def oracle_sample(inp, n_tokens):
    """Inputs restricted to the first n_tokens tokens (weights unchanged)."""
    sub = dict(inp)
    for key in ("x", "dY", "logits_in"):
        if key in sub:
            sub[key] = sub[key][:n_tokens]
    return sub


def run_oracle_step(w, f64, n_tokens):
    from oracle import moe_oracle_cpp as orc
    cap = orc.capacity_of(n_tokens, w.k, w.E) if w.capacity > 0 else 0
    t0 = time.perf_counter()
    fwd = orc.layer_forward(f64, w.k, cap)
    orc.layer_backward(f64, fwd)
    return time.perf_counter() - t0


def oracle_tokens(w, inp_f64, budget_s):
    """Tokens per oracle step so that one step costs about budget_s of CPU
    time: a 64-token calibration step, then proportional sizing (multiples of
    64, at least 64, at most T)."""
    t = run_oracle_step(w, oracle_sample(inp_f64, 64), 64)
    n = int(budget_s / max(t, 1e-6) * 64) // 64 * 64
    return max(64, min(w.T, n))


def cpu_baseline(w, inp, n_tokens=0, budget_s=20.0):
    from oracle import moe_oracle_cpp as orc
    f64 = orc.inputs_to_f64(inp)
    n = min(n_tokens, w.T) if n_tokens > 0 else oracle_tokens(w, f64, budget_s)
    t = run_oracle_step(w, oracle_sample(f64, n), n)
    return {"value": n / t, "unit": "tokens/s", "cores": orc.threads(), "kind": "oracle",
            "sample": f"{n} of {w.T} tokens of {w.name} (the first), forward+backward, the C++ fp64 oracle "
                      f"on {orc.threads()} host threads, one step of {t:.1f} s"}


def main_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    w = backward_workload(args.workload)
    inp = workloads.make_inputs(w)
    from oracle import moe_oracle_cpp as orc
    f64 = orc.inputs_to_f64(inp)
    nsteps = args.steps + args.warmup
    n = min(args.cpu_sample_tokens, w.T) if args.cpu_sample_tokens > 0 else \
        oracle_tokens(w, f64, REFERENCE_BUDGET_S / max(1, nsteps))
    sub = oracle_sample(f64, n)
    for _ in range(args.warmup):
        run_oracle_step(w, sub, n)
    times = [run_oracle_step(w, sub, n) for _ in range(args.steps)]
    total = sum(times)
    value = n * args.steps / total
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded SplitMix64/Box-Muller generator)",
        "config": {"workload": w.name, "T": w.T, "d": w.d, "E": w.E, "k": w.k, "H": w.H, "Hs": w.Hs,
                   "routing": w.routing, "capacity": w.capacity, "pass": "forward+backward",
                   "sample_tokens": n},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": orc.threads(), "kind": "oracle",
                         "sample": f"{n} of {w.T} tokens per step (the first), forward+backward, the C++ fp64 "
                                   f"oracle on {orc.threads()} host threads"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


# ------------------------------------------------------------------ our arm
def main_ours(args):
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl")

    import __graft_entry__
    # one build per node: local rank 0 compiles (if anything changed) while
    # the other ranks wait, then find it up to date
    if world > 1 and local != 0:
        dist.barrier()
    __graft_entry__.build()
    if world > 1 and local == 0:
        dist.barrier()
    from top_routing_grouped_moe_gb300 import _binding as B
    from top_routing_grouped_moe_gb300.layer import MoELayer

    w = backward_workload(args.workload)
    # every rank draws its own tokens (weak scaling); weights are the same
    seed = 20261202 + 7919 * rank
    inp = workloads.make_inputs(w, base=seed)
    dev = {}
    for key, v in inp.items():
        if key in ("bias", "logits_in"):
            dev[key] = torch.from_numpy(v).cuda()
        else:
            dev[key] = torch.from_numpy(v.view(np.int16)).cuda().view(torch.bfloat16)
    learned = w.routing == "learned"
    fused = args.path == "fused"
    # one layer per call sequence (same inputs, same results); the reported
    # path's layer is `layer`
    layers = {p: MoELayer(w.T, w.d, w.E, w.k, w.H, w.Hs, w.capacity, fused=(p == "fused"))
              for p in ("fused", "unfused")}
    layer = layers[args.path]
    L = layer
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    main_stream = torch.cuda.current_stream()
    T, d, E, k, H, Hs = w.T, w.d, w.E, w.k, w.H, w.Hs
    logits_in = dev.get("logits_in")

    def calls(lay):
        """The forward and the step of one layer: its C-ABI call sequence
        (MoELayer.forward / backward), on a given stream."""
        def forward(stream):
            lay.forward(dev["x"], dev, logits_in=logits_in, stream=stream)

        def step(stream):
            lay.forward(dev["x"], dev, logits_in=logits_in, stream=stream)
            lay.backward(dev["x"], dev["dY"], dev, learned_router=learned, stream=stream)
        return forward, step

    def forward_nosave(stream):
        """The forward alone as a forward-only pass runs it: a|u are not kept
        for a backward (the activation-recompute form of the forward)."""
        keep = layer.recompute
        layer.recompute = True
        try:
            layer.forward(dev["x"], dev, logits_in=logits_in, stream=stream)
        finally:
            layer.recompute = keep

    forward, step = calls(layer)
    other = "unfused" if fused else "fused"
    other_forward, other_step = calls(layers[other])

    for _ in range(max(3, args.warmup)):
        flush.fill_(1)
        step(main_stream)
        if not args.no_other_path:
            flush.fill_(1)
            other_step(main_stream)
    torch.cuda.synchronize()
    st = B.moe_device_status()
    if st != 0:
        raise RuntimeError(f"device status {st}: {B.status_string(st)}")
    R = int(layer.offsets[-1].item())

    # ---- eager steps (the calls issued one by one), timed by the library's
    # own event marks, L2 flushed before each: the eager step time and the
    # number of kernel launches per step
    eager_ms = []
    n_kernels = 0
    for i in range(args.steps):
        flush.fill_(i & 0xFF)
        with B.LaunchTimer(capacity=64, stream=main_stream) as tm:
            step(main_stream)
        torch.cuda.synchronize()
        lst = tm.launches()
        eager_ms.append(sum(ms for _, ms in lst))
        n_kernels = sum(1 for name, _ in lst if not name.startswith("memset"))
    eager_total = max_over_ranks([sum(eager_ms)], "cuda")[0]

    # ---- the step (and the forward alone) as CUDA-graph replays
    gstream = torch.cuda.Stream()
    graphs = {}
    graph_fns = [("step", step), ("forward", forward), ("forward_nosave", forward_nosave)]
    if not args.no_other_path:
        graph_fns += [("other_step", other_step), ("other_forward", other_forward)]
    for gname, fn in graph_fns:
        gstream.wait_stream(main_stream)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=gstream):
            fn(gstream)
        main_stream.wait_stream(gstream)
        graphs[gname] = g
    for g in graphs.values():
        for _ in range(3):
            flush.fill_(1)
            g.replay()
    torch.cuda.synchronize()
    st = B.moe_device_status()
    if st != 0:
        raise RuntimeError(f"device status {st} after graph replay: {B.status_string(st)}")

    def replay_ms(g, flush_l2=True):
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        for i in range(args.steps):
            if flush_l2:
                flush.fill_(1)
            ev[i][0].record()
            g.replay()
            ev[i][1].record()
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        return max_over_ranks([sum(a.elapsed_time(b) for a, b in ev)], "cuda")[0]

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    wall0 = time.perf_counter()
    graph_ms = replay_ms(graphs["step"])
    wall = time.perf_counter() - wall0
    fwd_ms = replay_ms(graphs["forward"])
    clocks = sampler.stop()
    nosave_ms = replay_ms(graphs["forward_nosave"])
    other_ms = replay_ms(graphs["other_step"]) if "other_step" in graphs else None
    other_fwd_ms = replay_ms(graphs["other_forward"]) if "other_forward" in graphs else None
    value = tokens_per_s(T, args.steps, world, graph_ms)
    fwd_value = tokens_per_s(T, args.steps, world, fwd_ms)

    def graph_launch_times(fn):
        """Every kernel launch of fn timed inside the timed region's form of
        it: fn captured in a CUDA graph with the library's timing marks (an
        event-record node before each launch), replayed args.steps times with
        L2 flushed before each.  {name: [ms of each launch]}"""
        tmr = B.LaunchTimer(capacity=64, stream=gstream)  # events created outside the capture
        gstream.wait_stream(main_stream)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=gstream):
            with tmr:
                fn(gstream)
        main_stream.wait_stream(gstream)
        for _ in range(3):
            flush.fill_(1)
            g.replay()
        times = {}
        for i in range(args.steps):
            flush.fill_(1)
            g.replay()
            torch.cuda.synchronize()
            for name, ms in tmr.launches():
                times.setdefault(name, []).append(ms)
        return times

    per_kernel = {name: {"launches_per_step": len(v) // args.steps, "ms": v}
                  for name, v in graph_launch_times(step).items()}
    timed_total = max_over_ranks([sum(sum(e["ms"]) for e in per_kernel.values())], "cuda")[0]
    # the smallest layer's working set fits in L2: its hot-L2 rate (replays
    # back to back, no flush) is reported beside the flushed one
    hot_l2 = None
    if w.name == "tiny":
        hot_ms, hot_fwd_ms = replay_ms(graphs["step"], False), replay_ms(graphs["forward"], False)
        hot_l2 = {"tokens_per_s": tokens_per_s(T, args.steps, world, hot_ms), "ms_per_step": hot_ms / args.steps,
                  "fwd_tokens_per_s": tokens_per_s(T, args.steps, world, hot_fwd_ms),
                  "fwd_ms_per_step": hot_fwd_ms / args.steps,
                  "note": "graph replays back to back without the L2 flush (working set resident in L2)"}

    def time_alone(fn):
        """mean ms of fn over args.steps calls after 3 warm-up calls, L2 flushed before each"""
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
        for i in range(args.steps + 3):
            if i >= 3:
                flush.fill_(1)
                ev[i - 3][0].record()
            fn()
            if i >= 3:
                ev[i - 3][1].record()
        torch.cuda.synchronize()
        return statistics.mean(a.elapsed_time(b) for a, b in ev)

    # calls of further rows of the hot path, timed alone (not part of the
    # configured step).  The router balance loss: loss, mean probabilities and
    # the logits gradient.
    lbl_logits = dev["logits_in"] if "logits_in" in dev else layer.logits
    lbl_out = torch.empty(1 + E + T * E, dtype=torch.float32, device="cuda")
    lbl_ms = time_alone(lambda: B.moe_router_balance_loss(
        lbl_logits, layer.counts_raw, T, E, k, 0.02, lbl_out[:1], lbl_out[1:1 + E], lbl_out[1 + E:],
        layer.ws, layer.ws_bytes))
    lbl_bytes = 2 * T * E * 4 + E * 8  # logits read, gradient written, counts and P
    # Activation recompute: the fp32 a|u rebuilt for the backward (gate/up GEMM
    # without the h store), written over the layer's saved copy (same values)
    if fused:
        rec_ms = time_alone(lambda: B.moe_grouped_swiglu_recompute_fused(
            dev["x"], layer.slot_of_row, layer.offsets, T, d, E, k, H, Hs, dev["W_g"], dev["W_u"],
            dev.get("Ws_g"), dev.get("Ws_u"), layer.au, layer.au_s))
    else:
        rec_ms = time_alone(lambda: B.moe_grouped_swiglu_recompute(
            layer.x_perm, layer.offsets, dev["x"], T, d, E, k, H, Hs, dev["W_g"], dev["W_u"],
            dev.get("Ws_g"), dev.get("Ws_u"), layer.au, layer.au_s))

    # ---- the MXFP8 forward (block-scaled E4M3 expert GEMMs): routing, the MX
    # permutation, the MX expert MLP and the combine, as a graph replay; the
    # weights and the shared expert's input are quantized once, before
    mx_fwd = None
    if d % 128 == 0 and Hs > 0:
        u8 = lambda n: torch.empty(n, dtype=torch.uint8, device="cuda")  # noqa: E731
        i32 = lambda n: torch.empty(n, dtype=torch.int32, device="cuda")  # noqa: E731
        mrows = B.moe_mxfp8_rows(T, E, k)
        sb = B.moe_mxfp8_scales_bytes
        mxb = {"off": i32(E + 1), "row": i32(T * k), "sor": i32(mrows), "cr": i32(E), "c": i32(E), "o0": i32(E + 1),
               "xc": u8(mrows * d), "xs": u8(sb(mrows, d)), "hc": u8(mrows * H), "hs": u8(sb(mrows, H)),
               "gu_c": u8(E * 2 * H * d), "gu_s": u8(sb(E * 2 * H, d)), "d_c": u8(E * d * H), "d_s": u8(sb(E * d, H)),
               "sgu_c": u8(2 * Hs * d), "sgu_s": u8(sb(2 * Hs, d)), "sd_c": u8(d * Hs), "sd_s": u8(sb(d, Hs)),
               "xsc": u8(T * d), "xss": u8(sb(T, d)), "hsc": u8(T * Hs), "hss": u8(sb(T, Hs)),
               "o": torch.empty(mrows, d, dtype=torch.float16, device="cuda"),
               "s": torch.empty(T, d, dtype=torch.float16, device="cuda"),
               "y": torch.empty(T, d, dtype=torch.bfloat16, device="cuda")}
        B.moe_mxfp8_quantize_gate_up(dev["W_g"], dev["W_u"], E, H, d, mxb["gu_c"], mxb["gu_s"])
        B.moe_mxfp8_quantize(dev["W_d"], E * d, H, mxb["d_c"], mxb["d_s"])
        B.moe_mxfp8_quantize_gate_up(dev["Ws_g"], dev["Ws_u"], 1, Hs, d, mxb["sgu_c"], mxb["sgu_s"])
        B.moe_mxfp8_quantize(dev["Ws_d"], d, Hs, mxb["sd_c"], mxb["sd_s"])

        def mx_forward(stream):
            x = dev["x"]
            B.moe_route_topk(x, dev.get("W_r"), dev.get("bias"), dev.get("logits_in"), T, d, E, k,
                             L.logits if learned else None, L.idx, L.gates, L.ws, L.ws_bytes, stream)
            B.moe_permute_mxfp8(x, L.idx, T, d, E, k, L.capacity, mxb["cr"], mxb["c"], mxb["o0"], mxb["off"],
                                mxb["row"], mxb["sor"], mxb["xc"], mxb["xs"], L.ws, L.ws_bytes, stream)
            B.moe_mxfp8_quantize(x, T, d, mxb["xsc"], mxb["xss"], stream)
            B.moe_grouped_swiglu_mxfp8(mxb["xc"], mxb["xs"], mxb["off"], mxb["c"], mxb["xsc"], mxb["xss"], T, d, E,
                                       k, H, Hs, mxb["gu_c"], mxb["gu_s"], mxb["d_c"], mxb["d_s"], mxb["sgu_c"],
                                       mxb["sgu_s"], mxb["sd_c"], mxb["sd_s"], mxb["hc"], mxb["hs"], mxb["hsc"],
                                       mxb["hss"], mxb["o"], mxb["s"], stream)
            B.moe_unpermute_combine_mxfp8(mxb["o"], mxb["s"], L.gates, mxb["row"], T, d, E, k, mxb["y"], stream)

        for _ in range(3):
            flush.fill_(1)
            mx_forward(main_stream)
        torch.cuda.synchronize()
        st = B.moe_device_status()
        if st != 0:
            raise RuntimeError(f"device status {st} in the MXFP8 forward: {B.status_string(st)}")
        mx_kernels = graph_launch_times(mx_forward)
        gstream.wait_stream(main_stream)
        gmx = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gmx, stream=gstream):
            mx_forward(gstream)
        main_stream.wait_stream(gstream)
        for _ in range(3):
            flush.fill_(1)
            gmx.replay()
        mx_ms = replay_ms(gmx)
        mx_fwd = {"tokens_per_s": tokens_per_s(T, args.steps, world, mx_ms), "ms_per_step": mx_ms / args.steps,
                  "kernels": {n: round(statistics.mean(v) * len(v) / args.steps, 4) for n, v in mx_kernels.items()},
                  "note": "forward with MXFP8 (E4M3, E8M0 per 32) expert and shared-expert GEMMs on the tensor "
                          "cores; routing, x quantized inside the permutation, combine; weights quantized once, "
                          "outside the timed region; graph replay, L2 flushed before each"}

    # ---- rooflines: measured burst peaks (kernels timed inside a step of a
    # few milliseconds)
    peaks = {}
    pk = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(pk):
        peaks = json.load(open(pk))
    tensor_peak = peaks.get("bf16_tflops") or 1900.0
    hbm_peak = peaks.get("hbm_gbs") or 6800.0
    peak_src = "measured" if peaks else "fallback"
    work = kernel_work(w, R, fused)
    issued = issued_mma_flops(w, R)
    step_eager = eager_total / args.steps
    step_timed = timed_total / args.steps
    kernels = {}
    for name, e in per_kernel.items():
        mean = statistics.mean(e["ms"])
        row = {"launches_per_step": e["launches_per_step"], "ms_per_launch": round(mean, 4),
               "share": round(mean * e["launches_per_step"] / step_timed, 4)}
        if name in work:
            row.update(kernel_roofline(work[name], mean, tensor_peak, hbm_peak))
            with_issued(row, name, issued, mean, tensor_peak)
        kernels[name] = row
    dom = max((n for n in kernels if n in work), key=lambda n: kernels[n]["share"])
    roof = dict(kernel_roofline(work[dom], kernels[dom]["ms_per_launch"], tensor_peak, hbm_peak))
    with_issued(roof, dom, issued, kernels[dom]["ms_per_launch"], tensor_peak)
    roof.update({"kernel": dom, "share_of_step": kernels[dom]["share"],
                 "traffic": profiled_traffic(w.name, dom),
                 "traffic_unit": "bytes per launch (ncu dram read + write)",
                 "peak_source": f"{peak_src} burst ({'bf16 cuBLAS' if roof['bound'] == 'tensor' else 'copy'})"})
    ffl, bfl = gemm_flops(w, R)
    rec_work = work["gemm_gate_up_recompute_gather" if fused else "gemm_gate_up_recompute"]
    if mx_fwd is not None:
        fp8_peak = 2.0 * tensor_peak  # the fp8 dense tensor rate is twice bf16's (nominal ratio)
        mx_fwd["rooflines"] = {}
        for name in ("gemm_mx_gate_up_swiglu", "gemm_mx_down", "perm_scatter_mx"):
            if name in mx_fwd["kernels"]:
                mx_fwd["rooflines"][name] = dict(kernel_roofline(work[name], mx_fwd["kernels"][name], fp8_peak,
                                                                 hbm_peak), ms=mx_fwd["kernels"][name])
        mx_fwd["fp8_peak_source"] = f"{peak_src} bf16 burst x 2 (nominal fp8 / bf16 ratio)"

    # ---- e2e through the public layer API with host buffers
    e2e = None
    if not args.no_e2e:
        pin = {}
        for key in ("x", "dY"):
            pin[key] = torch.from_numpy(inp[key].view(np.int16)).view(torch.bfloat16).pin_memory()
        if "logits_in" in inp:
            pin["logits_in"] = torch.from_numpy(inp["logits_in"]).pin_memory()
        y_host = torch.empty(T, d, dtype=torch.bfloat16).pin_memory()
        dx_host = torch.empty(T, d, dtype=torch.bfloat16).pin_memory()
        h2d = pin["x"].numel() * 2 + pin["dY"].numel() * 2 + (pin["logits_in"].numel() * 4 if "logits_in" in pin else 0)
        d2h = 2 * T * d * 2

        # The loop a training job runs: every step uploads its x and dY from
        # pinned host memory and downloads y and dx, through the layer API.
        # Inputs are double-buffered: step i+1's upload runs (on its own
        # stream) beside step i's backward, y's download beside the backward,
        # dx's beside the next forward.  Events order every reuse: a buffer is
        # refilled only after the backward that read it, and y / dx are
        # overwritten only after their downloads.
        up, down = torch.cuda.Stream(), torch.cuda.Stream()
        xin = [torch.empty_like(dev["x"]) for _ in range(2)]
        dyin = [torch.empty_like(dev["dY"]) for _ in range(2)]
        lin = [torch.empty_like(dev["logits_in"]) for _ in range(2)] if "logits_in" in dev else None

        def upload(b, after):
            with torch.cuda.stream(up):
                if after is not None:
                    up.wait_event(after)
                xin[b].copy_(pin["x"], non_blocking=True)
                if lin is not None:
                    lin[b].copy_(pin["logits_in"], non_blocking=True)
                dyin[b].copy_(pin["dY"], non_blocking=True)
                return up.record_event()

        def e2e_run(n):
            main = torch.cuda.current_stream()
            ready = upload(0, None)
            freed = [None, None]
            y_copied = dx_copied = None
            p = dict(dev)
            for i in range(n):
                b = i & 1
                main.wait_event(ready)
                if y_copied is not None:
                    main.wait_event(y_copied)
                layer.forward(xin[b], p, logits_in=lin[b] if lin is not None else None)
                fwd_done = main.record_event()
                with torch.cuda.stream(down):
                    down.wait_event(fwd_done)
                    y_host.copy_(layer.y, non_blocking=True)
                    y_copied = down.record_event()
                if i + 1 < n:
                    ready = upload(1 - b, freed[1 - b])
                if dx_copied is not None:
                    main.wait_event(dx_copied)
                layer.backward(xin[b], dyin[b], p, learned_router=learned)
                freed[b] = main.record_event()
                with torch.cuda.stream(down):
                    down.wait_event(freed[b])
                    dx_host.copy_(layer.dx, non_blocking=True)
                    dx_copied = down.record_event()
            main.synchronize()
            down.synchronize()
            up.synchronize()

        e2e_run(3)
        if world > 1:
            dist.barrier()
        t0 = time.perf_counter()
        e2e_run(args.steps)
        el = max_over_ranks([time.perf_counter() - t0], "cuda")[0]
        e2e = {"value": tokens_per_s(T, args.steps, world, el * 1000.0), "unit": "tokens/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, inp, args.cpu_sample_tokens)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": max(3, args.warmup), "ms_per_step": graph_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded SplitMix64/Box-Muller generator)",
            "config": {"workload": w.name, "T": T, "d": d, "E": E, "k": k, "H": H, "Hs": Hs,
                       "routing": w.routing, "capacity": w.capacity, "pass": "forward+backward",
                       "l2": "flushed before every step (256 MB write)", "parallelism": f"replicas x{world}",
                       "timing": "value / fwd_tokens_per_s: the C-ABI calls of the step / of the forward "
                                 "captured once in a CUDA graph and replayed; kernels: every launch of the "
                                 "step, timed by event-record nodes the library puts before each launch in a "
                                 "graph of the step, replayed the same way"},
            "fwd_tokens_per_s": fwd_value,
            "path": args.path,
            "other_path": None if other_ms is None else {
                "path": other, "tokens_per_s": tokens_per_s(T, args.steps, world, other_ms),
                "ms_per_step": other_ms / args.steps,
                "fwd_tokens_per_s": tokens_per_s(T, args.steps, world, other_fwd_ms),
                "fwd_ms_per_step": other_fwd_ms / args.steps,
                "note": "the same step through the other call sequence (identical results); "
                        "graph replay, L2 flushed before each"},
            "mxfp8_forward": mx_fwd,
            "fwd_ms_per_step": fwd_ms / args.steps,
            "fwd_nosave": {"tokens_per_s": tokens_per_s(T, args.steps, world, nosave_ms),
                           "ms_per_step": nosave_ms / args.steps,
                           "gemm_tflops": ffl / (nosave_ms / args.steps / 1000.0) / 1e12,
                           "note": "the forward as a forward-only pass: a|u not kept for a backward; graph "
                                   "replay, L2 flushed before each"},
            "hot_l2": hot_l2,
            "eager": {"value": tokens_per_s(T, args.steps, world, eager_total), "ms_per_step": step_eager},
            "gemm_tflops_fwd_bwd": (ffl + bfl) / (graph_ms / args.steps / 1000.0) / 1e12,
            # the forward alone (configurations whose pass is the forward)
            "gemm_tflops_fwd": ffl / (fwd_ms / args.steps / 1000.0) / 1e12,
            "gemm_frac_bf16_fwd": round(ffl / (fwd_ms / args.steps / 1000.0) / 1e12 / tensor_peak, 4),
            "gemm_frac_bf16_fwd_bwd": round((ffl + bfl) / (graph_ms / args.steps / 1000.0) / 1e12 / tensor_peak, 4),
            "roofline": roof,
            "kernels": dict(sorted(kernels.items(), key=lambda kv: -kv[1]["share"])),
            "extra_calls": {
                "moe_router_balance_loss": {
                    "ms": round(lbl_ms, 4), "gbs": round(lbl_bytes / (lbl_ms / 1000.0) / 1e9, 1),
                    "frac_hbm": round(lbl_bytes / (lbl_ms / 1000.0) / 1e9 / hbm_peak, 3),
                    "note": "one kernel after a 4-byte memset; timed alone, not part of the step"},
                "moe_grouped_swiglu_recompute": dict(
                    kernel_roofline(rec_work, rec_ms, tensor_peak, hbm_peak), ms=round(rec_ms, 4),
                    note="one GEMM launch; timed alone, not part of the step")},
            "clocks": clocks,
            "gpu_launches": n_kernels * args.steps,
            "e2e": e2e,
            "cpu_baseline": cpu,
            "wall_s_timed_region": wall,
        }
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()
    return 0


def main():
    args = parse()
    if args.impl == "reference":
        return main_reference(args)
    return main_ours(args)


if __name__ == "__main__":
    sys.exit(main())
