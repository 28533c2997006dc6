"""Benchmark of the forward-convolution library on GB300.

Default workload: the video-VAE Convolution3D layer (conv3d, fp16 storage,
fp32 accumulation, N=1, IC=128, 5 frames of 128x240, OC=128, k=3, pad 1,
stride 1, bias; NCDHW x, OIDHW weights packed inside the call), the largest
of the five layer shapes and the one the pages time (SeedVR2's VAE decoder,
git.erdda.com/Tencent/ncnn/discussions/7001). One step is one forward call
through the C ABI (gbconv_conv3d_fwd) with inputs resident in HBM; steps
rotate over copies of x and y larger than L2 (129 MB), so no step finds its
operands there. The line also carries the per-layer TFLOP/s, GB/s and
roofline fraction of all five layer shapes (`--workload` picks any of them
as the headline), an end-to-end number with host buffers, and the CPU oracle
timed on the host cores as a baseline.

Multi-GPU: each rank runs an independent replica of the workload on its own
GPU (the layer is one problem; no data exchange), barrier + synchronize
around the timed region, max time over ranks; value = FLOP of all ranks / that
time ("scaling": "weak").

`--impl reference` times the fp64 CPU oracle (the only reference
implementation: the pages ship no runnable code) on the same layer, on the
host cores.
"""
import argparse
import dataclasses
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synthetic  # noqa: E402

METRIC = ("conv TFLOP/s and % of roofline per layer shape at 1 GB300 "
          "(vs CPU oracle)")
WORKLOADS = {"detection_stem": 2, "tiny": 1, "text_line_batch": 3,
             "wide_dense_f16": 4, "video_vae_conv3d_f16": 5}
# Variants of a layer shape: (layer, fields changed, name suffix). The fused
# 2x2 max pool of the stem, the video-VAE conv3d with causal frame padding,
# and the two tensor-core layers with channels-last activations (x read in
# place, no layout pass: the layer-chaining case).
VARIANTS = {"detection_stem_maxpool": (2, {"pool": True}, "+maxpool2x2"),
            "video_vae_conv3d_f16_causal": (5, {"tpad": 1}, "+causal_frames"),
            "wide_dense_f16_channels_last": (4, {"cl": True}, "+channels_last"),
            "video_vae_conv3d_f16_channels_last": (5, {"cl": True}, "+channels_last"),
            "text_line_batch_exact_fp32": (3, {}, "+exact_fp32_cuda_cores")}
# Variants that force an algorithm: the fp32 layer on the CUDA cores (exact
# fp32 FMAs) instead of the tensor cores' three TF32 products.
VARIANT_ALGO = {"text_line_batch_exact_fp32": "IGEMM_FFMA"}


def workload_algo(gb, name):
    """The algorithm a workload forces (ALGO_AUTO unless it names one)."""
    return getattr(gb, "ALGO_" + VARIANT_ALGO[name]) if name in VARIANT_ALGO else gb.ALGO_AUTO


def workload_layer(name):
    if name in WORKLOADS:
        return synthetic.LAYERS[WORKLOADS[name]]
    idx, kw, suffix = VARIANTS[name]
    base = synthetic.LAYERS[idx]
    return dataclasses.replace(base, name=base.name + suffix, **kw)
DEFAULT_WORKLOAD = "video_vae_conv3d_f16"


def device_x(L, inp):
    """x as the call takes it: NC(D)HW, or channels-last for a `cl` layer."""
    return np.ascontiguousarray(np.moveaxis(inp.x, 1, -1)) if L.cl else inp.x
FLUSH_BYTES = 256 << 20
SM_COUNT_FALLBACK = 152
FP32_LANES_PER_SM = 128


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        p = json.load(open(path))
        return {"hbm_gbs": float(p["hbm_gbs"]),
                "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained",
                                                     p["bf16_tflops"])),
                "sm_max_mhz": float(p.get("sm_max_mhz", 2070.0)),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0,
            "bf16_tflops_sustained": 1700.0, "sm_max_mhz": 2070.0,
            "source": "fallback"}


def fp32_peak_tflops(pk, sms):
    """CUDA-core FFMA peak: SMs x 128 lanes x 2 FLOP x max SM clock."""
    return sms * FP32_LANES_PER_SM * 2 * pk["sm_max_mhz"] * 1e6 / 1e12


def fp32_split_peak_tflops(pk):
    """fp32 convolution FLOP rate of three TF32 products on the tensor cores:
    the dense TF32 rate (half the bf16 rate: 1.1 vs 2.25 PFLOP/s nominal)
    divided by the three products each fp32 product costs."""
    return pk["bf16_tflops"] / 2 / 3


# ------------------------------------------------------------- replicas
def max_over_ranks(ms, world, device="cpu"):
    """The slowest rank's time (ms) for the timed region: every rank runs
    its own replica of the layer, so the job takes as long as the slowest."""
    if world <= 1:
        return float(ms)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(flop_per_step, steps, world, total_ms):
    """Whole-job throughput: the FLOP of all ranks' steps over the slowest
    rank's time."""
    return flop_per_step * steps * world / (total_ms * 1e-3) / 1e12


# --------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clock/throttle samples every 100 ms while running. It runs
    over the whole bench (the timed region of a short run lasts milliseconds,
    below the sampler's period); `summary` reports the samples taken while
    the GPU drew power well above idle, i.e. under this run's load."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,"
         "clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.idx = device_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), "--query-gpu=" + self.Q,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, note=None):
        rows, mx = [], None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        for ln in self.lines:
            f = [v.strip() for v in ln.split(",")]
            if len(f) < 8:
                continue
            try:
                sm, mx, pw = float(f[1]), float(f[2]), float(f[3])
            except ValueError:
                continue
            rows.append((sm, pw, {n for n, v in zip(names, f[4:8]) if v.lower() == "active"}))
        # under load: power at least idle + 30% of the range seen
        if rows:
            p_lo, p_hi = min(r[1] for r in rows), max(r[1] for r in rows)
            load = [r for r in rows if r[1] >= p_lo + 0.3 * (p_hi - p_lo)] or rows
        else:
            load = []
        reasons = set().union(*[r[2] for r in load]) if load else set()
        out = {"sm_mhz": statistics.median(r[0] for r in load) if load else None,
               "sm_max_mhz": mx, "reasons": sorted(reasons),
               "samples": len(rows), "samples_under_load": len(load),
               "power_w_max": max((r[1] for r in rows), default=None)}
        if note:
            out["window"] = note
        return out


# --------------------------------------------------------- traffic table
def recorded_traffic(kernel_file, key):
    """DRAM bytes per launch from the committed ncu summary, or None when
    that kernel's source changed since the counters were taken."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    src = os.path.join(ROOT, "implicit_gemm_convolution_conv_gb300", "csrc",
                       kernel_file)
    if not os.path.exists(path) or not os.path.exists(src):
        return None
    sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    for line in open(path):
        f = line.split()
        if len(f) == 3 and not line.startswith("#") and f[0] == key:
            return int(f[1]) if f[2] == sha else None
    return None


# ------------------------------------------------------------- rotation
ROTATE_BYTES = 256 << 20     # > 2 x L2: a set is cold when it comes round again


GRAPH_CALLS = 64     # calls per captured graph, at least (see Rotation.graphs)


def graph_plan(steps, copies):
    """How Rotation.graphs splits `steps` calls over `copies` buffer copies:
    (calls per graph, replays of it, calls in a last shorter graph). A graph
    holds whole rounds over the copies and at least GRAPH_CALLS calls, or all
    the steps when there are fewer."""
    per = min(steps, copies * -(-GRAPH_CALLS // copies))
    full, tail = divmod(steps, per)
    return per, full, tail


class Rotation:
    """R copies of the layer's input/output buffers used in turn, so that no
    step finds its x or y in L2 (R x set bytes >= 256 MiB); steps are
    recorded into CUDA graphs of back-to-back forward calls."""

    def __init__(self, torch, conv, rotate=True):
        self.torch = torch
        x = conv.x
        set_bytes = (x.numel() + conv.y.numel()) * x.element_size()
        r = max(1, -(-ROTATE_BYTES // set_bytes)) if rotate else 1
        self.resident = r > 64 or not rotate
        r = min(r, 64)
        self.convs = [conv] + [conv.with_input(x.clone()) for _ in range(r - 1)]
        self.i = 0
        self.l2_note = (f"inputs rotated over {r} copies of x and y "
                        f"({r * set_bytes / 2**20:.0f} MiB > L2)"
                        if not self.resident else
                        f"{r} cop{'y' if r == 1 else 'ies'} of a {set_bytes} B "
                        "layer: L2-resident")

    def eager_step(self):
        self.convs[self.i % len(self.convs)]()
        self.i += 1

    def graphs(self, steps):
        """CUDA graphs whose replay runs exactly `steps` calls in turn. A graph
        holds a whole number of rounds over the copies and at least
        GRAPH_CALLS calls (fewer only when `steps` is smaller): consecutive
        calls inside a graph overlap through programmatic dependent launch,
        while a boundary between two replays costs a graph launch, which one
        graph per round (a single call for an L2-resident layer) would add
        to every few calls."""
        torch = self.torch
        r = len(self.convs)
        per, full, tail = graph_plan(steps, r)
        out = []
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        def capture(n):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                for j in range(n):
                    self.convs[j % r]()
            return g
        if full:
            g = capture(per)
            out += [g] * full
        if tail:
            out.append(capture(tail))
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        return out


# ---------------------------------------------------------------- ours
def run_ours(args):
    import torch
    import torch.distributed as dist
    import implicit_gemm_convolution_conv_gb300 as gb
    from implicit_gemm_convolution_conv_gb300.torch_ops import Conv, to_device

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    props = torch.cuda.get_device_properties(dev)
    sms = props.multi_processor_count or SM_COUNT_FALLBACK
    pk = peaks()
    stream = torch.cuda.current_stream()
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    def timed_calls(conv, reps, warm, do_flush=True):
        for _ in range(warm):
            conv()
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True),
                torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        for e0, e1 in evs:
            if do_flush:
                flush.zero_()
            e0.record(stream)
            conv()
            e1.record(stream)
        torch.cuda.synchronize()
        return [e0.elapsed_time(e1) for e0, e1 in evs]

    clk = ClockSampler(local).__enter__()
    L = workload_layer(args.workload)
    inp = synthetic.make_inputs(L)
    x, w = to_device(device_x(L, inp), L.dtype, dev), to_device(inp.w, L.dtype, dev)
    b = torch.from_numpy(inp.b).to(dev)
    algo = workload_algo(gb, args.workload)
    conv = Conv(x, w, b, L.stride, L.pad, L.relu, tpad=L.tpad, pool=L.pool, channels_last=L.cl, algo=algo)
    # the tensor-core GEMM's x layout pass (when x is not read in place)
    # shares one launch with the weight pack
    launches = {gb.ALGO_DIRECT: 1, gb.ALGO_DIRECT_TC: 1, gb.ALGO_IGEMM_FFMA: 2,
                gb.ALGO_IGEMM_TC: 2}[conv.algo]
    x_in_place = L.cl and L.dtype != "f32" and L.C % 8 == 0
    rot = Rotation(torch, conv)

    # warm-up, then exactly K timed steps between barriers
    for _ in range(args.warmup):
        rot.eager_step()
    barrier()
    graphs = rot.graphs(args.steps)
    # each distinct graph once, untimed: its first replay uploads it
    for g in {id(g): g for g in graphs}.values():
        g.replay()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    t_wall = time.perf_counter()
    e0.record(stream)
    for g in graphs:
        g.replay()
    e1.record(stream)
    barrier()
    t_wall = time.perf_counter() - t_wall
    total_ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    flops = L.flops()
    value = job_tflops(flops, args.steps, world, total_ms)
    avg_s = total_ms / args.steps * 1e-3
    iso = timed_calls(conv, 50, 3)
    line = None
    if rank == 0:
        stem = L.ndim == 2 and L.C <= 4 and L.k == 3 and L.stride in (1, 2)
        # stems of at most 65,536 outputs (no pool) run one thread per output
        tiny = stem and not L.pool and int(np.prod(L.y_shape())) <= 1 << 16
        kernel, kfile = {gb.ALGO_DIRECT: (("direct_tiny_kernel" if tiny else "direct_stem_kernel"), "direct_stem.cu")
                         if stem else ("direct_conv_kernel", "direct.cu"),
                         gb.ALGO_DIRECT_TC: ("stem_tf32_kernel", "stem_tf32.cuh"),
                         gb.ALGO_IGEMM_FFMA: (("igemm_ffma_kernel" if L.C % 16 or L.cl else
                                               "igemm_ffma_cp_kernel" if L.dtype == "f32" else
                                               "igemm_ffma2_kernel"), "igemm_ffma.cu"),
                         gb.ALGO_IGEMM_TC: ("igemm_tc_kernel", "igemm_tc.cu")}[conv.algo]
        kernel_key = f"{kernel}:{L.name}"
        if conv.algo in (gb.ALGO_DIRECT, gb.ALGO_DIRECT_TC):
            achieved = L.compulsory_bytes() / avg_s / 1e9
            roof = {"bound": "hbm", "achieved": round(achieved, 1),
                    "peak": pk["hbm_gbs"], "unit": "GB/s",
                    "frac": round(achieved / pk["hbm_gbs"], 4),
                    "algorithmic_bytes_per_launch": L.compulsory_bytes(),
                    "peak_source": pk["source"] + " hbm_gbs (burst copy)"}
        elif conv.algo == gb.ALGO_IGEMM_FFMA:
            p32 = fp32_peak_tflops(pk, sms)
            achieved = L.flops() / avg_s / 1e12
            roof = {"bound": "alu", "achieved": round(achieved, 3),
                    "peak": round(p32, 2), "unit": "TFLOP/s",
                    "frac": round(achieved / p32, 4),
                    "algorithmic_flops_per_launch": L.flops(),
                    "peak_source": "derived: SMs x 128 FP32 lanes x 2 x max SM clock"}
        elif L.dtype == "f32":
            # fp32 on the tensor cores: three TF32 products per fp32 product
            pt = fp32_split_peak_tflops(pk)
            achieved = L.flops() / avg_s / 1e12
            roof = {"bound": "tensor", "achieved": round(achieved, 2),
                    "peak": round(pt, 1), "unit": "TFLOP/s",
                    "frac": round(achieved / pt, 4),
                    "algorithmic_flops_per_launch": L.flops(),
                    "peak_source": pk["source"] + " bf16_tflops / 2 (TF32 rate) / 3 (products per fp32 product)"}
        else:
            achieved = L.flops() / avg_s / 1e12
            roof = {"bound": "tensor", "achieved": round(achieved, 2),
                    "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                    "frac": round(achieved / pk["bf16_tflops"], 4),
                    "algorithmic_flops_per_launch": L.flops(),
                    "peak_source": pk["source"] + " bf16_tflops (burst; fp16 dense rate equals bf16)"}
        roof["traffic"] = recorded_traffic(kfile, kernel_key)
        roof["kernel"] = kernel
        roof["timed"] = ("one call = one launch" if launches == 1 else
                         f"one call = {launches} launches (weight pack"
                         + ("" if x_in_place or conv.algo != gb.ALGO_IGEMM_TC
                            else " and x layout pass in one grid")
                         + ", GEMM); times are per call")
        line = {
            "metric": METRIC, "value": round(value, 3), "unit": "TFLOP/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(total_ms / args.steps, 6),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32" if L.dtype == "f32" else L.dtype,
            "data": "synthetic (seeded; shapes of the pages' layers)",
            "config": {"workload": L.name, "N": L.N, "C": L.C, "D": L.D,
                       "H": L.H, "W": L.W, "OC": L.OC, "k": L.k,
                       "pad": L.pad, "stride": L.stride, "relu": L.relu,
                       "algo": gb.algo_name(conv.algo),
                       "l2": rot.l2_note,
                       "timing": "CUDA graph of back-to-back forward calls "
                                 "replayed; events around all K steps",
                       "parallelism": f"replicas x{world}"},
            "roofline": roof,
            "gpu_launches": launches * args.steps,
            "wall_s_timed_region": round(t_wall, 4),
            "latency_us_isolated_call": round(statistics.median(iso) * 1e3, 3),
            "latency_us_isolated_call_p10": quantile_us(iso, 0.1),
            "latency_us_isolated_call_p90": quantile_us(iso, 0.9),
        }
    barrier()

    if rank == 0:
        # end to end: pinned host buffers, H2D of x, w, b and D2H of y inside
        # the timed region, through the same C-ABI call. Consecutive steps
        # rotate over three streams, each with its own device buffers (x, w,
        # b, y, workspace), so one step's D2H overlaps the next steps' H2D
        # and calls; every step still copies all its inputs in and its output
        # out. Each stream's step (three copies in, the call, one copy out)
        # is captured once into a CUDA graph and replayed, so the host issues
        # one launch per step instead of five calls (page 2,
        # m.demingchina.com/news/41165: capture and replay hides the host's
        # per-call launch cost).
        hx = torch.from_numpy(np.ascontiguousarray(device_x(L, inp))).pin_memory()
        hw = torch.from_numpy(np.ascontiguousarray(inp.w)).pin_memory()
        hb = torch.from_numpy(inp.b).pin_memory()
        reps = min(args.steps, 200)
        n_pipe = 3
        pipes = []
        for _ in range(n_pipe):
            xj, wj, bj = torch.empty_like(x), torch.empty_like(w), torch.empty_like(b)
            xj.copy_(x)
            wj.copy_(w)
            bj.copy_(b)
            cj = Conv(xj, wj, bj, L.stride, L.pad, L.relu, tpad=L.tpad, pool=L.pool, channels_last=L.cl,
                      algo=algo)
            hyj = torch.empty(cj.y.shape, dtype=cj.y.dtype).pin_memory()
            pipes.append((torch.cuda.Stream(), xj, wj, bj, cj, hyj))
        torch.cuda.synchronize()
        cap = torch.cuda.Stream()
        cap.wait_stream(torch.cuda.current_stream())
        step_graphs = []
        for sj, xj, wj, bj, cj, hyj in pipes:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=cap):
                xj.copy_(hx, non_blocking=True)
                wj.copy_(hw, non_blocking=True)
                bj.copy_(hb, non_blocking=True)
                cj()
                hyj.copy_(cj.y, non_blocking=True)
            step_graphs.append(g)
        torch.cuda.current_stream().wait_stream(cap)
        torch.cuda.synchronize()

        def e2e_step(i):
            sj = pipes[i % n_pipe][0]
            with torch.cuda.stream(sj):
                step_graphs[i % n_pipe].replay()
        for i in range(3 * n_pipe):
            e2e_step(i)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for pj in pipes:
            pj[0].wait_stream(stream)
        for i in range(reps):
            e2e_step(i)
        for pj in pipes:
            stream.wait_stream(pj[0])
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = e0.elapsed_time(e1) / reps
        hy = pipes[0][5]
        # The host link's floor for this step on this machine: the same copies
        # alone (H2D of x, w, b and D2H of y on two streams at once), no call.
        s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
        _, x0, w0, b0, c0, hy0 = pipes[0]

        def copies():
            s_in.wait_stream(stream)
            s_out.wait_stream(stream)
            with torch.cuda.stream(s_in):
                x0.copy_(hx, non_blocking=True)
                w0.copy_(hw, non_blocking=True)
                b0.copy_(hb, non_blocking=True)
            with torch.cuda.stream(s_out):
                hy0.copy_(c0.y, non_blocking=True)
            stream.wait_stream(s_in)
            stream.wait_stream(s_out)
        for _ in range(3):
            copies()
        torch.cuda.synchronize()
        n_copy = 20
        e0.record(stream)
        for _ in range(n_copy):
            copies()
        e1.record(stream)
        torch.cuda.synchronize()
        copy_ms = e0.elapsed_time(e1) / n_copy
        line["e2e"] = {"value": round(flops / (e2e_ms * 1e-3) / 1e12, 4),
                       "unit": "TFLOP/s",
                       "h2d_bytes_per_step": hx.numel() * hx.element_size() +
                       hw.numel() * hw.element_size() + hb.numel() * 4,
                       "d2h_bytes_per_step": hy.numel() * hy.element_size(),
                       "ms_per_step": round(e2e_ms, 5),
                       "copies_only_ms_per_step": round(copy_ms, 5),
                       "streams": n_pipe,
                       "issue": "one CUDA graph per stream: H2D x, w, b; the C-ABI call; D2H y"}
        if not args.skip_layers:
            line["per_layer"] = per_layer(gb, Conv, to_device, torch, dev,
                                          timed_calls, pk, sms)
        clk.__exit__()
        line["clocks"] = clk.summary("whole bench run: warm-up, timed steps, isolated calls, "
                                     "end-to-end and per-layer timing (samples every 100 ms)")
        if not args.skip_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(L, inp, budget_s=args.cpu_seconds)
        print(json.dumps(line), flush=True)
    else:
        clk.__exit__()
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


def quantile_us(ms, f):
    """The f-quantile (linear interpolation between order statistics) of
    event times given in ms, in us."""
    q = sorted(ms)
    i = f * (len(q) - 1)
    lo = int(i)
    hi = min(lo + 1, len(q) - 1)
    return round((q[lo] + (q[hi] - q[lo]) * (i - lo)) * 1e3, 3)


def per_layer(gb, Conv, to_device, torch, dev, timed_calls, pk, sms):
    """TFLOP/s, GB/s and roofline fraction of every layer shape: average
    call time of back-to-back calls on rotated buffers (graph replay), with
    OIHW weights packed inside the call and with pre-packed weights; plus
    the isolated latency of one eager call after an L2 flush, and the
    back-to-back time with L2-resident buffers."""
    out = []
    p32 = fp32_peak_tflops(pk, sms)
    layers = [(idx, L, gb.ALGO_AUTO) for idx, L in sorted(synthetic.LAYERS.items())] + [
        (VARIANTS[v][0], workload_layer(v), workload_algo(gb, v)) for v in sorted(VARIANTS)]
    for idx, L, algo in layers:
        inp = synthetic.make_inputs(L)
        x, w = to_device(device_x(L, inp), L.dtype, dev), to_device(inp.w, L.dtype, dev)
        b = torch.from_numpy(inp.b).to(dev)
        rec = {"layer": L.name, "flop": L.flops(),
               "bytes": L.compulsory_bytes()}
        pc = p32 if L.dtype == "f32" else pk["bf16_tflops"]
        pc_split = fp32_split_peak_tflops(pk)
        t_c = L.flops() / (pc * 1e12)
        t_m = L.compulsory_bytes() / (pk["hbm_gbs"] * 1e9)
        t_ideal = max(t_c, t_m)
        for prepack in (False, True):
            conv = Conv(x, w, b, L.stride, L.pad, L.relu, prepack=prepack, tpad=L.tpad, pool=L.pool,
                        channels_last=L.cl, algo=algo)
            rot = Rotation(torch, conv)
            calls = 200 if idx <= 3 else (100 if idx == 4 else 40)
            for _ in range(3):
                rot.eager_step()
            gs = rot.graphs(calls)
            for g in {id(g): g for g in gs}.values():
                g.replay()              # upload, untimed
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for g in gs:
                g.replay()
            e1.record()
            torch.cuda.synchronize()
            s = e0.elapsed_time(e1) / calls * 1e-3
            warm_rot = Rotation(torch, conv, rotate=False)
            gw = warm_rot.graphs(calls)
            for g in {id(g): g for g in gw}.values():
                g.replay()
            e0.record()
            for g in gw:
                g.replay()
            e1.record()
            torch.cuda.synchronize()
            s_warm = e0.elapsed_time(e1) / calls * 1e-3
            iso = timed_calls(conv, 20, 2)
            key = "prepacked" if prepack else "oihw"
            # fp32 on the tensor cores (three TF32 products) is held to that
            # path's own compute ceiling; the CUDA-core FP32 peak stays as a
            # second figure
            split = L.dtype == "f32" and conv.algo == gb.ALGO_IGEMM_TC
            t_c_run = L.flops() / (pc_split * 1e12) if split else t_c
            rec[key] = {
                "algo": gb.algo_name(conv.algo),
                "us_per_call": round(s * 1e6, 3),
                "tflops": round(L.flops() / s / 1e12, 3),
                "gbs": round(L.compulsory_bytes() / s / 1e9, 1),
                "roofline_frac": round(max(t_c_run, t_m) / s, 4),
                "roofline_frac_at_3.35TBs": round(max(t_c_run, L.compulsory_bytes() / 3.35e12) / s, 4),
                "bound": (("tensor" if split or L.dtype != "f32" else "fp32")
                          if t_c_run > t_m else "hbm"),
                **({"roofline_frac_vs_cuda_core_fp32_peak": round(t_ideal / s, 4)} if split else {}),
                "compute_peak_tflops": round(pc_split if split else pc, 1),
                "l2": rot.l2_note,
                "us_per_call_l2_resident": round(s_warm * 1e6, 3),
                "us_isolated_call_median": round(statistics.median(iso) * 1e3, 3),
                "us_isolated_call_p10": quantile_us(iso, 0.1),
                "us_isolated_call_p90": quantile_us(iso, 0.9),
            }
            del conv, rot, warm_rot, gs, gw
        out.append(rec)
        del x, w, b
    return out


def oracle_layer(oracle, L, inp):
    """The oracle's whole result for a layer (conv, then the 2x2 max pool
    when the layer has one)."""
    y = oracle.conv(inp.x, inp.w, inp.b, L.stride, L.pad, L.relu, L.dtype, tpad=L.tpad)
    return oracle.maxpool2(y) if L.pool else y


def cpu_baseline(L, inp, budget_s=10.0):
    """The oracle as it stands on the host cores, on the whole layer when
    one call fits the budget, else on a sample of outputs."""
    import oracle
    threads = oracle.threads()
    t0 = time.perf_counter()
    oracle_layer(oracle, L, inp)
    one = time.perf_counter() - t0
    if one <= budget_s / 2 or L.pool:
        reps, t0 = 0, time.perf_counter()
        while time.perf_counter() - t0 < budget_s and reps < 100000:
            oracle_layer(oracle, L, inp)
            reps += 1
        dt = time.perf_counter() - t0
        flop = L.flops() * reps
        sample = f"whole layer, {reps} calls"
    else:
        total = int(np.prod(L.y_shape()))
        n = max(1000, int(total * (budget_s / 2) / one))
        idx = np.random.Generator(np.random.PCG64(1)).integers(0, total, n)
        t0 = time.perf_counter()
        oracle.conv_at(inp.x, inp.w, inp.b, idx, L.stride, L.pad, L.relu,
                       L.dtype, tpad=L.tpad)
        dt = time.perf_counter() - t0
        flop = L.flops() * n / total
        sample = f"{n} of {total} outputs"
    return {"value": round(flop / dt / 1e12, 6), "unit": "TFLOP/s",
            "cores": threads, "kind": "oracle", "sample": sample,
            "seconds": round(dt, 3)}


# ----------------------------------------------------------- reference
# Reference-arm steps: layers up to REF_WHOLE_FLOP run whole; larger ones
# time a seeded sample of about REF_STEP_FLOP of their outputs per step, so
# that the default K and W stay within minutes on the host.
REF_WHOLE_FLOP = 5e9
REF_STEP_FLOP = 2e9


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    L = workload_layer(args.workload)
    inp = synthetic.make_inputs(L)
    import oracle
    threads = oracle.threads()
    total = int(np.prod(L.y_shape()))
    if L.flops() <= REF_WHOLE_FLOP or L.pool:
        # a step is one whole-layer oracle call
        step = lambda: oracle_layer(oracle, L, inp)
        step_flop, sample = L.flops(), f"whole layer per step, {args.steps} steps"
    else:
        # a step is the same seeded sample of outputs, about REF_STEP_FLOP
        # of the layer's work, computed one by one
        n = max(1000, int(total * REF_STEP_FLOP / L.flops()))
        idx = np.random.Generator(np.random.PCG64(2)).integers(0, total, n)
        step = lambda: oracle.conv_at(inp.x, inp.w, inp.b, idx, L.stride, L.pad, L.relu,
                                      L.dtype, tpad=L.tpad)
        step_flop = L.flops() * n / total
        sample = f"{n} of {total} outputs per step (seeded), {args.steps} steps"
    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t0
    value = step_flop * args.steps / dt / 1e12
    line = {"metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s",
            "n_gpus": int(os.environ.get("WORLD_SIZE", "1")),
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(dt / args.steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic (seeded; shapes of the pages' layers)",
            "config": {"workload": L.name, "parallelism": "host cores"},
            "impl": "reference",
            "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s",
                             "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 6), "unit": "TFLOP/s",
                    "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS) + sorted(VARIANTS), default=DEFAULT_WORKLOAD)
    ap.add_argument("--skip-layers", action="store_true")
    ap.add_argument("--skip-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        if args.steps > 50:
            args.steps = 50       # keep the CPU run to a few minutes
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
