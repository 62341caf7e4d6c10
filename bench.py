"""Benchmark of the NVFP4 decode-step weight stream on GB300.

Workload (default): the ~31B-shaped decoder stack, 60 layers x {fused QKV
[8192, 5376], o_proj [5376, 4096], fused gate+up [43008, 5376], down
[5376, 21504]} in NVFP4 (13,934,592,000 bytes of weights, far larger than
L2), one bf16 token per projection, all 240 projections streamed in order on
one stream per step: aq_decode_step_weights (one GEMV launch per fused
projection, programmatic dependent launch between them) captured once in a
CUDA graph and replayed.  Weights are seeded synthetic N(0, 0.02^2) with
0.1% x20 outliers, quantised on the GPU by the library before timing.

Metric: algorithmic HBM GB/s of the step (0.5625 B per weight element + 4 B
per-tensor scale + activations in + outputs out) and ms per step.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl aq|reference]
                    [--workload 31b|1b] [--layers L] [--m M] [--no-extras]
                    [--batch-sweep] [--bf16-lm-head] [--load-time]

One JSON line is printed by rank 0.  With N > 1 (torchrun) every rank runs
an independent replica on its own GPU (the path has no exchange step).
``--layers`` streams only the first L layers (a small case for profilers).
"""
import argparse
import hashlib
import json
import os
import platform
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "NVFP4 decode GEMV HBM GB/s (% of 8 TB/s); ms per 31B-shaped step weight stream"
NOMINAL_HBM_GBS = 8000.0  # the 8 TB/s denominator the metric names

# DRAM bytes of one layer's GEMV launches (dram__bytes_read.sum +
# dram__bytes_write.sum summed over the layer's four launches in one ncu
# capture), keyed by the workload and the sha1 of the GEMV kernel sources the
# capture was taken on; when they change the figure no longer applies (null).
NCU_TRAFFIC = {
    # the four launches of one layer (layer 3 of an 8-layer stream, so no
    # weight of the layer can still sit in L2 from an earlier step), m = 1,
    # one-token kernel form, captured without cache flushing so the L2
    # prefetch of the next projection counts where it is issued: reads
    # 19,480,320 + 15,461,888 + 144,582,656 + 67,476,736, writes 227,328 +
    # 102,912 + 492,032 + 238,848 (the committed ncu summary of that capture)
    ("gemma4-31b-shaped decode-step weight stream", 1, "9615d4ee255ae3c2bd9bdb6ff4c8ba8b51741a51"): 248062720,
}


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=("aq", "reference"), default="aq")
    p.add_argument("--m", type=int, default=1, help="tokens per projection")
    p.add_argument("--workload", choices=("31b", "1b"), default="31b")
    p.add_argument("--layers", type=int, default=0,
                   help="stream only the first L layers (0: all of the workload's layers)")
    p.add_argument("--batch-sweep", action="store_true",
                   help="time the ~31B-shaped fused gate+up and down weights at M in "
                        "{1, 2, 4, 8, 16, 32, 64} on every path instead of the step")
    p.add_argument("--sweep-m", type=str, default="",
                   help="comma-separated subset of the sweep's M values (profiling)")
    p.add_argument("--sweep-proj", choices=("both", "gate_up", "down"), default="both")
    p.add_argument("--kernel", choices=("regdecode", "tcgen05", "mma"), default="regdecode",
                   help="GEMV kernel of the timed step (regdecode: the library's default "
                        "for m <= 16; the other one is timed among the extras)")
    p.add_argument("--bf16-lm-head", action="store_true",
                   help="time only the bf16 GEMV on the ~31B tied lm_head [262144, 5376], m = 1")
    p.add_argument("--profile-case", choices=("gemv", "load"), default="",
                   help="a few calls on one ~31B projection, for profilers (not a timing)")
    p.add_argument("--profile-proj", type=int, choices=(0, 1, 2, 3), default=2)
    p.add_argument("--small-configs", action="store_true",
                   help="1B-shaped single projections (fused QKV, MLP) per call, L2-cold and warm")
    p.add_argument("--load-time", action="store_true",
                   help="time only the load-time kernels (reconstruct + quantise, and "
                        "quantise alone) on the 1B MLP shapes and the ~31B gate+up")
    p.add_argument("--no-extras", action="store_true",
                   help="skip the eager / no-PDL / end-to-end / CPU-baseline legs")
    return p.parse_args()


def workload(name):
    from nvfp4_block_scaled_aq_gb300 import inputs
    if name == "31b":
        return "gemma4-31b-shaped decode-step weight stream", inputs.LAYER_31B, inputs.LAYERS_31B
    return "gemma3-1b-shaped decode-step weight stream", inputs.LAYER_1B, inputs.LAYERS_1B


def algorithmic_bytes(shapes, layers, m):
    """Bytes one step must move at minimum: NVFP4 weights (packed nibbles +
    one E4M3 scale per 16 elements = 0.5625 B/element), the fp32 per-tensor
    scale, the bf16 activations read and the bf16 outputs written."""
    per_layer = 0
    for n, k in shapes:
        per_layer += n * k // 2 + n * k // 16 + 4 + 2 * m * k + 2 * m * n
    return per_layer * layers


def load_time_bytes(n, k, r, fused):
    """Algorithmic bytes of one load-time call on an [n, k] weight: the bf16
    weight (W0 for the fused form) read once, the packed nibbles, one E4M3
    scale per 16 elements and the fp32 g_dec written; the fused form also
    reads s (fp32 per row) and U, V (bf16, rank r)."""
    byts = n * k * 2 + n * k // 2 + n * k // 16 + 4
    if fused:
        byts += 4 * n + 2 * (n + k) * r
    return byts


def weight_bytes(shapes, layers):
    return sum(n * k // 2 + n * k // 16 for n, k in shapes) * layers


# ------------------------------------------------------------ distributed

class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist
            backend = "nccl" if self._cuda() else "gloo"
            dist.init_process_group(backend)
            self.pg = dist

    @staticmethod
    def _cuda():
        import torch
        return torch.cuda.is_available()

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, v):
        if not self.pg:
            return v
        import torch
        t = torch.tensor([v], dtype=torch.float64,
                         device="cuda" if self._cuda() else "cpu")
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


# ------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.samples = []
        self.error = None
        self.proc = None
        self.t0 = self.t1 = None
        cmd = ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
               "-lms", "100"]
        sel = self._selector(device_index)
        if sel:
            cmd += ["-i", sel]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError as e:
            self.error = str(e)

    @staticmethod
    def _selector(idx):
        try:
            import torch
            u = str(torch.cuda.get_device_properties(idx).uuid)
            return u if u.startswith("GPU-") else "GPU-" + u
        except Exception:
            return None

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 8:
                self.samples.append((time.time(), parts))

    def window(self, t0, t1):
        self.t0, self.t1 = t0, t1

    def stop(self):
        if self.proc:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [],
                    "note": self.error or "no nvidia-smi samples"}
        inside = [p for t, p in self.samples
                  if self.t0 is None or (self.t0 - 0.1 <= t <= self.t1 + 0.1)]
        if not inside:  # timed region shorter than the sampling period
            mid = 0.5 * (self.t0 + self.t1)
            inside = [min(self.samples, key=lambda s: abs(s[0] - mid))[1]]
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(p[0]) for p in inside if num(p[0]) is not None]
        mx = [num(p[1]) for p in inside if num(p[1]) is not None]
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({nm for p in inside for nm, v in zip(names, p[4:8])
                          if v.strip().lower() == "active"})
        pw = [num(p[2]) for p in inside if num(p[2]) is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(inside), "power_w_max": max(pw) if pw else None}


# ------------------------------------------------------------ the aq arm

class Stack:
    """All projections of the workload resident in HBM, plus one
    activation buffer and one output buffer sliced per projection."""

    def __init__(self, shapes, layers, m, device, seed=0):
        import torch
        from nvfp4_block_scaled_aq_gb300 import aq, inputs
        self.shapes, self.layers, self.m = shapes, layers, m
        qws = torch.zeros(aq.quantize_workspace_bytes(), dtype=torch.uint8, device=device)
        self.weights = []
        for layer in range(layers):
            for p, (n, k) in enumerate(shapes):
                W = inputs.weight(n, k, seed=inputs.seed_of(seed, layer, p), device=device)
                w = aq.Nvfp4Weight.empty(n, k, device=device)
                aq.quantize(W, w, qws)
                del W
                self.weights.append(w)
        x_elems = [m * k for _ in range(layers) for (n, k) in shapes]
        y_elems = [m * n for _ in range(layers) for (n, k) in shapes]
        self.x_all = torch.empty(sum(x_elems), dtype=torch.bfloat16, device=device)
        self.y_all = torch.empty(sum(y_elems), dtype=torch.bfloat16, device=device)
        self.xs, self.ys = [], []
        xo = yo = 0
        for i, (xe, ye) in enumerate(zip(x_elems, y_elems)):
            n, k = shapes[i % len(shapes)]
            self.xs.append(self.x_all[xo:xo + xe].view(m, k))
            self.ys.append(self.y_all[yo:yo + ye].view(m, n))
            xo += xe
            yo += ye
        for i, x in enumerate(self.xs):
            layer, p = divmod(i, len(shapes))
            x.copy_(inputs.tokens(m, x.shape[1], seed=inputs.seed_of(seed + 1, layer, p),
                                  device=device))
        ws_bytes = max(aq.gemv_workspace_bytes(n, k, m) for n, k in shapes)
        self.ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=device)
        self.args = aq.StepArgs(self.weights, self.xs, self.ys)
        self.plan = aq.StepPlan(self.weights, self.xs, self.ys)
        self.plan_ws = self.plan.workspace()
        torch.cuda.synchronize()
        st = aq.poll_device_status()
        if st != aq.OK:
            raise RuntimeError("quantisation reported %s: %s" % (st, aq.last_error()))

    @property
    def launches(self):
        return len(self.weights)


def capture(stack, flags, stream):
    import torch
    from nvfp4_block_scaled_aq_gb300 import aq
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        aq.decode_step(stack.args, stack.ws, flags=flags, stream=stream)
        stream.synchronize()
        with torch.cuda.graph(g, stream=stream):
            aq.decode_step(stack.args, stack.ws, flags=flags, stream=stream)
    torch.cuda.synchronize()
    return g


def time_region(run_step, steps, warmup, stream, dist, sampler=None):
    """Seconds for `steps` steps: barrier + synchronize on both sides, CUDA
    events recorded on the launching stream; max over ranks."""
    import torch
    for _ in range(warmup):
        run_step()
    torch.cuda.synchronize()
    dist.barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    t0 = time.time()
    e0.record(stream)
    for _ in range(steps):
        run_step()
    e1.record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    dist.barrier()
    if sampler:
        sampler.window(t0, t1)
    return dist.max(e0.elapsed_time(e1) / 1e3)


def bf16_lm_head_leg(stream, dist, a, device):
    """The bf16 GEMV on the ~31B tied lm_head [262144, 5376] at m = 1
    (2.82 GB, far larger than L2): a CUDA graph of 8 PDL-chained calls,
    event-timed on the launching stream."""
    import torch
    from nvfp4_block_scaled_aq_gb300 import aq, inputs
    n, k = inputs.LM_HEAD_31B
    W = inputs.weight(n, k, seed=inputs.seed_of(9000), device=device, outliers=False)
    x = inputs.tokens(1, k, seed=inputs.seed_of(9001), device=device)
    y = torch.empty((1, n), dtype=torch.bfloat16, device=device)
    ws = torch.zeros(aq.gemv_bf16_workspace_bytes(n, k, 1), dtype=torch.uint8, device=device)
    calls = 8
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        aq.gemv_bf16(W, x, y, ws, flags=aq.STEP_PDL, stream=stream)
        stream.synchronize()
        with torch.cuda.graph(g, stream=stream):
            for _ in range(calls):
                aq.gemv_bf16(W, x, y, ws, flags=aq.STEP_PDL, stream=stream)
    torch.cuda.synchronize()

    def run():
        with torch.cuda.stream(stream):
            g.replay()
    reps = max(3, a.steps // 10)
    secs = time_region(run, reps, a.warmup, stream, dist) / (reps * calls)
    torch.cuda.synchronize()
    del g
    byts = 2 * n * k + 2 * k + 2 * n
    peak, _ = load_peaks()
    return {"shape": [n, k], "m": 1, "us_per_call": round(secs * 1e6, 2),
            "GBps": round(byts / secs / 1e9, 1), "frac_of_peak": round(byts / secs / 1e9 / peak, 4),
            "kernel": "gemv_bf16_kernel<1>, 8 PDL-chained calls per CUDA graph"}


def epilogue_leg(stream, dist, a, device):
    """The GEMV's epilogue variants on the ~31B fused gate+up [43008, 5376]
    at m = 1 -- plain, runtime low-rank (rank 4), fused activation h =
    gelu(gate) * up -- each as a graph of 8 PDL-chained calls alternating
    two weight copies (260 MB, twice L2), event-timed on the launching
    stream."""
    import torch
    from nvfp4_block_scaled_aq_gb300 import aq, inputs
    n, k = inputs.LAYER_31B[2]
    r = 4
    ws_w = []
    for c in range(2):
        W = inputs.weight(n, k, seed=inputs.seed_of(9100 + c), device=device)
        w = aq.Nvfp4Weight.empty(n, k, device=device)
        aq.quantize(W, w, torch.zeros(aq.quantize_workspace_bytes(), dtype=torch.uint8,
                                      device=device))
        ws_w.append(w)
        del W
    g = torch.Generator(device="cpu").manual_seed(9102)
    s = torch.exp(0.1 * torch.randn(n, generator=g)).to(torch.float32).to(device)
    U = (0.01 * torch.randn((n, r), generator=g)).to(torch.bfloat16).to(device)
    V = (0.01 * torch.randn((k, r), generator=g)).to(torch.bfloat16).to(device)
    x = inputs.tokens(1, k, seed=inputs.seed_of(9103), device=device)
    y = torch.empty((1, n), dtype=torch.bfloat16, device=device)
    ws = torch.zeros(aq.gemv_lowrank_workspace_bytes(n, k, 1, r), dtype=torch.uint8, device=device)
    calls = 8

    def graph(fn):
        torch.cuda.synchronize()
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            fn(0)
            stream.synchronize()
            with torch.cuda.graph(gr, stream=stream):
                for i in range(calls):
                    fn(i & 1)
        torch.cuda.synchronize()

        def run():
            with torch.cuda.stream(stream):
                gr.replay()
        reps = max(3, a.steps // 10)
        secs = time_region(run, reps, a.warmup, stream, dist) / (reps * calls)
        del gr
        return secs

    t_lr = graph(lambda i: aq.gemv_lowrank(ws_w[i], s, U, V, x, y, ws, flags=aq.STEP_PDL,
                                           stream=stream))
    t_plain = graph(lambda i: aq.decode_step(aq.StepArgs([ws_w[i]], [x], [y]), ws,
                                             flags=aq.STEP_PDL | aq.STEP_REGDECODE,
                                             stream=stream))
    h = torch.empty((1, n // 2), dtype=torch.bfloat16, device=device)
    t_glu = graph(lambda i: aq.gemv_glu(ws_w[i], x, h, ws, flags=aq.STEP_PDL, stream=stream))
    byts = 0.5625 * n * k + 4 + 2 * k + 2 * n
    return {"shape": [n, k], "m": 1,
            "plain_us_per_call": round(t_plain * 1e6, 2),
            "plain_GBps": round(byts / t_plain / 1e9, 1),
            "lowrank_r4_us_per_call": round(t_lr * 1e6, 2),
            "glu_us_per_call": round(t_glu * 1e6, 2),
            "kernels": "gemv_kernel<1, plain | low-rank (after vx_kernel) | GLU epilogue>"}


def small_gemv_timing(n, k, copies, pdl, stream, dist, a, device):
    """Microseconds per call of the m = 1 NVFP4 GEMV on [n, k]: a CUDA graph
    of calls over `copies` seeded weights in turn (one copy: the same weight
    every call, L2-warm), with or without programmatic dependent launch
    between the calls; event-timed on the launching stream."""
    import torch
    from nvfp4_block_scaled_aq_gb300 import aq, inputs
    qws = torch.zeros(aq.quantize_workspace_bytes(), dtype=torch.uint8, device=device)
    ws_w = []
    for c in range(copies):
        W = inputs.weight(n, k, seed=inputs.seed_of(9700 + c), device=device)
        w = aq.Nvfp4Weight.empty(n, k, device=device)
        aq.quantize(W, w, qws)
        ws_w.append(w)
        del W
    x = inputs.tokens(1, k, seed=inputs.seed_of(9701), device=device)
    y = torch.empty((1, n), dtype=torch.bfloat16, device=device)
    ws = torch.zeros(aq.gemv_workspace_bytes(n, k, 1), dtype=torch.uint8, device=device)
    calls = max(copies, 64)
    flags = aq.STEP_REGDECODE | (aq.STEP_PDL if pdl else 0)
    args = [aq.StepArgs([w], [x], [y]) for w in ws_w]
    torch.cuda.synchronize()
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        aq.decode_step(args[0], ws, flags=flags, stream=stream)
        stream.synchronize()
        with torch.cuda.graph(gr, stream=stream):
            for i in range(calls):
                aq.decode_step(args[i % copies], ws, flags=flags, stream=stream)
    torch.cuda.synchronize()

    def run():
        with torch.cuda.stream(stream):
            gr.replay()
    reps = max(5, a.steps // 10)
    secs = time_region(run, reps, a.warmup, stream, dist) / (reps * calls)
    del gr, ws_w
    torch.cuda.synchronize()
    return secs


def run_small_configs(a, dist):
    """The 1B-shaped single projections at m = 1: the fused QKV [1536,
    1152] and the MLP's fused gate+up [13824, 1152] and down [1152, 6912].
    Per call: L2-cold (a graph over seeded weight copies that together
    exceed twice L2, in turn), chained with programmatic dependent launch
    and stream-ordered without it, and L2-warm (one weight, every call).
    GB/s of algorithmic bytes (0.5625 B per weight element + 4 + 2k + 2n)."""
    import torch
    from nvfp4_block_scaled_aq_gb300 import aq, inputs
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(dist.local)
    device = torch.device("cuda", dist.local)
    stream = torch.cuda.Stream(device)
    peak, src = load_peaks()
    rows = []
    for name, (n, k) in (("fused_qkv", inputs.LAYER_1B[0]), ("fused_gate_up", inputs.LAYER_1B[2]),
                         ("down", inputs.LAYER_1B[3])):
        byts = n * k // 2 + n * k // 16 + 4 + 2 * k + 2 * n
        copies = -(-(2 * 129 * 10**6) // (n * k // 2 + n * k // 16))
        row = {"name": name, "shape": [n, k], "m": 1, "algorithmic_bytes": byts, "cold_copies": copies}
        for label, cp, pdl in (("cold_pdl", copies, True), ("cold_no_pdl", copies, False),
                               ("warm_pdl", 1, True)):
            secs = small_gemv_timing(n, k, cp, pdl, stream, dist, a, device)
            row[label] = {"us_per_call": round(secs * 1e6, 3), "GBps": round(byts / secs / 1e9, 1),
                          "frac_of_peak": round(byts / secs / 1e9 / peak, 4)}
        rows.append(row)
    st = aq.poll_device_status()
    if st != aq.OK:
        raise RuntimeError("device status %d: %s" % (st, aq.last_error()))
    if dist.rank == 0:
        print(json.dumps({"metric": "1B-shaped single-projection NVFP4 GEMV, us per call and GB/s",
                          "value": rows[0]["cold_pdl"]["us_per_call"], "unit": "us per call (fused QKV, cold, PDL)",
                          "n_gpus": dist.world, "higher_is_better": False,
                          "data": "synthetic (seeded N(0,0.02^2) weights with 0.1% x20 outliers, N(0,1) tokens)",
                          "config": {"workload": "1B-shaped fused QKV, gate+up and down at m = 1",
                                     "l2": "cold legs rotate over weight copies exceeding twice L2"},
                          "hbm_peak_gbs": peak, "hbm_peak_source": src, "projections": rows}), flush=True)


def run_profile_case(a, dist):
    """A small case for profilers: four calls on one ~31B-shaped projection
    (--profile-proj: 0 fused QKV, 1 o_proj, 2 fused gate+up, 3 down),
    alternating two seeded weight copies so no call finds its weights in L2.
    --profile-case gemv: aq_gemv_nvfp4 with --m tokens on the register-decode
    kernel (--kernel regdecode) or the block-scaled MMA path (--kernel mma);
    --profile-case load: aq_reconstruct_quantize_nvfp4 of a rank-4 theta
    bundle.  Prints one JSON line with the device status; not a timing."""
    import torch
    from nvfp4_block_scaled_aq_gb300 import aq, inputs
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(dist.local)
    device = torch.device("cuda", dist.local)
    n, k = inputs.LAYER_31B[a.profile_proj]
    qws = torch.zeros(aq.quantize_workspace_bytes(), dtype=torch.uint8, device=device)
    if a.profile_case == "load":
        th = inputs.theta(n, k, 4, seed=inputs.seed_of(9800), device=device)
        w = aq.Nvfp4Weight.empty(n, k, device=device)
        for _ in range(4):
            aq.reconstruct_quantize(th.W0, th.s, th.U, th.V, w, qws)
    else:
        ws_w = []
        for c in range(2):
            W = inputs.weight(n, k, seed=inputs.seed_of(0, c, a.profile_proj), device=device)
            w = aq.Nvfp4Weight.empty(n, k, device=device)
            aq.quantize(W, w, qws)
            ws_w.append(w)
            del W
        x = inputs.tokens(a.m, k, seed=inputs.seed_of(1, 0, a.profile_proj), device=device)
        y = torch.empty((a.m, n), dtype=torch.bfloat16, device=device)
        ws = torch.zeros(aq.gemv_workspace_bytes(n, k, a.m), dtype=torch.uint8, device=device)
        path = aq.PATH_MMA if a.kernel == "mma" else aq.PATH_GEMV_REGDECODE
        for i in range(4):
            aq.gemv(ws_w[i % 2], x, y, ws, path=path)
    torch.cuda.synchronize()
    st = aq.poll_device_status()
    if dist.rank == 0:
        print(json.dumps({"profile_case": a.profile_case, "shape": [n, k], "m": a.m,
                          "kernel": a.kernel, "status": st}), flush=True)


def kernel_sha():
    h = hashlib.sha1()
    for name in ("gemv_core.cuh", "gemv.cu"):
        h.update(open(os.path.join(ROOT, "nvfp4_block_scaled_aq_gb300", "csrc", name), "rb").read())
    return h.hexdigest()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return float(pk["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def host_cpu():
    """(model name, usable host cores) of the machine the oracle runs on."""
    model = platform.machine()
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.split(":")[0].strip() in ("Model name", "Vendor ID") and ":" in line:
                model = line.split(":", 1)[1].strip()
                if line.startswith("Model name"):
                    break
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        cores = len(os.sched_getaffinity(0))
    except AttributeError:
        cores = os.cpu_count() or 1
    return model, cores


def oracle_rows(shapes, m, seed=0, max_rows=8192):
    """Layer 0's projections quantised by the oracle (seeded like the GPU
    workload, drawn on the CPU): (packed, scales, g_dec, x, rows, k) each."""
    import oracle
    from nvfp4_block_scaled_aq_gb300 import inputs
    prepared = []
    for p, (n, k) in enumerate(shapes):
        rows = min(n, max_rows)
        W = inputs.bits_u16(inputs.weight(rows, k, seed=inputs.seed_of(seed, 0, p)))
        x = inputs.bits_u16(inputs.tokens(m, k, seed=inputs.seed_of(seed + 1, 0, p)))
        packed, scales, ge, gd = oracle.quantize(W)
        prepared.append((packed, scales, gd, x, rows, k))
    return prepared


def oracle_gemv_leg(prepared, m, threads, budget_s):
    """The oracle's fp64 GEMV, as it stands, over 64-row chunks of the
    prepared projections (each projection gets an equal share of the time
    budget), on `threads` host threads at once (ctypes releases the GIL for
    the C call, so the threads run on separate cores).  Returns (bytes,
    wall seconds, rows)."""
    import concurrent.futures as cf
    import threading
    import numpy as np
    import oracle
    done = [0.0, 0]
    lock = threading.Lock()
    wall = 0.0
    for packed, scales, gd, x, rows, k in prepared:
        chunks = iter(range(0, rows, 64))
        deadline = [None]

        def worker():
            while True:
                with lock:
                    if time.perf_counter() > deadline[0]:
                        return
                    r0 = next(chunks, None)
                if r0 is None:
                    return
                r1 = min(rows, r0 + 64)
                oracle.gemv(packed, scales, gd, x, rows=np.arange(r0, r1))
                with lock:
                    done[0] += (r1 - r0) * (k // 2 + k // 16) + 2 * m * (r1 - r0)
                    done[1] += r1 - r0
        t = time.perf_counter()
        deadline[0] = t + budget_s / len(prepared)
        with cf.ThreadPoolExecutor(max_workers=threads) as ex:
            for f in [ex.submit(worker) for _ in range(threads)]:
                f.result()
        wall += time.perf_counter() - t
        done[0] += 2 * m * k + 4
    return done[0], wall, done[1]


def cpu_baseline(shapes, m, budget_s=12.0, seed=0):
    """The oracle's fp64 GEMV, as it stands, on the host: rows of layer 0's
    projections until the time budget is spent, first on one core, then on
    every host core at once.  Returns GB/s of algorithmic bytes for the
    all-cores leg, with the one-core leg beside it."""
    prepared = oracle_rows(shapes, m, seed)
    model, cores = host_cpu()
    b1, s1, r1 = oracle_gemv_leg(prepared, m, 1, budget_s / 3)
    bn, sn, rn = oracle_gemv_leg(prepared, m, cores, budget_s * 2 / 3)
    total_rows = sum(n for n, _ in shapes)
    return {"value": bn / sn / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "cpu": model,
            "sample": "%d rows of layer-0 projections (of %d rows x 60 layers), m=%d, "
                      "fp64 accumulation, %d threads (one per host core)" % (rn, total_rows, m, cores),
            "seconds": round(sn, 3),
            "single_thread": {"value": b1 / s1 / 1e9, "unit": "GB/s", "cores": 1,
                              "sample": "%d rows" % r1, "seconds": round(s1, 3)}}


def run_aq(a, dist):
    import torch
    from nvfp4_block_scaled_aq_gb300 import aq
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(dist.local)
    device = torch.device("cuda", dist.local)
    name, shapes, layers = workload(a.workload)
    layer_traffic = NCU_TRAFFIC.get((name, a.m, kernel_sha()))
    if a.layers:
        layers = min(layers, a.layers)
        name += " (first %d layers)" % layers
    stack = Stack(shapes, layers, a.m, device)
    step_bytes = algorithmic_bytes(shapes, layers, a.m)
    stream = torch.cuda.Stream(device)

    def replay(graph):
        def run():
            with torch.cuda.stream(stream):  # replay on the stream the events time
                graph.replay()
        return run

    def persistent():
        aq.step_run(stack.plan, stack.plan_ws, stream=stream)

    # the timed path: one GEMV launch per projection (PDL), captured in a
    # graph, on the kernel chosen by --kernel (the library's default unless
    # asked otherwise: fixed, so a profiler's launch list sees the same legs)
    flags = {"regdecode": aq.STEP_REGDECODE, "tcgen05": aq.STEP_TCGEN05}
    if a.kernel == "mma":  # the block-scaled MMA path, on request only
        flags["mma"] = aq.STEP_MMA
    kernel = a.kernel
    kflag = flags[kernel]
    g_pdl = capture(stack, aq.STEP_PDL | kflag, stream)
    sampler = ClockSampler(dist.local) if dist.rank == 0 else None
    time.sleep(0.3 if sampler else 0)
    secs = time_region(replay(g_pdl), a.steps, a.warmup, stream, dist, sampler)
    if sampler:
        sampler.stop()
    ms = secs / a.steps * 1e3
    value = dist.world * step_bytes * a.steps / secs / 1e9

    extras = {"kernel": kernel}
    e2e = None
    if not a.no_extras:
        kernel_ms = {kernel: ms}
        for kname, fl in flags.items():
            if kname != kernel:
                g = capture(stack, aq.STEP_PDL | fl, stream)
                kernel_ms[kname] = time_region(replay(g), a.steps, a.warmup, stream, dist) \
                    / a.steps * 1e3
                del g
        extras["graph_pdl_ms_per_step_by_kernel"] = {k: round(v, 4) for k, v in kernel_ms.items()}
        extras["persistent_step_run_ms_per_step"] = round(
            time_region(persistent, a.steps, a.warmup, stream, dist) / a.steps * 1e3, 4)
        g_nopdl = capture(stack, kflag, stream)
        extras["per_projection_graph_no_pdl_ms_per_step"] = round(
            time_region(replay(g_nopdl), a.steps, a.warmup, stream, dist) / a.steps * 1e3, 4)
        del g_nopdl

        def eager():
            aq.decode_step(stack.args, stack.ws, flags=aq.STEP_PDL | kflag, stream=stream)
        with torch.cuda.stream(stream):
            extras["per_projection_eager_pdl_ms_per_step"] = round(
                time_region(eager, a.steps, a.warmup, stream, dist) / a.steps * 1e3, 4)

        # end to end through the C ABI: pinned host activations in, outputs out
        x_host = torch.empty(stack.x_all.numel(), dtype=torch.bfloat16, pin_memory=True)
        x_host.copy_(stack.x_all)
        y_host = torch.empty(stack.y_all.numel(), dtype=torch.bfloat16, pin_memory=True)

        def e2e_step():
            with torch.cuda.stream(stream):
                stack.x_all.copy_(x_host, non_blocking=True)
                g_pdl.replay()
                y_host.copy_(stack.y_all, non_blocking=True)
        e2e_secs = time_region(e2e_step, a.steps, a.warmup, stream, dist)
        e2e = {"value": round(dist.world * step_bytes * a.steps / e2e_secs / 1e9, 2),
               "unit": "GB/s",
               "ms_per_step": round(e2e_secs / a.steps * 1e3, 4),
               "h2d_bytes_per_step": stack.x_all.numel() * 2,
               "d2h_bytes_per_step": stack.y_all.numel() * 2,
               "path": "aq_decode_step_weights graph replay, pinned host buffers copied "
                       "in and out inside the timed region"}
    del g_pdl
    if not a.no_extras and a.workload == "31b":
        extras["bf16_lm_head"] = bf16_lm_head_leg(stream, dist, a, device)
        extras["gate_up_epilogues"] = epilogue_leg(stream, dist, a, device)

    st = aq.poll_device_status()
    if st != aq.OK:
        raise RuntimeError("device status %d after timing: %s" % (st, aq.last_error()))

    peak, peak_kind = load_peaks()
    # the step is stack.launches GEMV launches; with PDL they overlap, so the
    # average launch is the step's bytes and time divided by the launch count
    launch_bytes = step_bytes / stack.launches
    launch_s = secs / a.steps / stack.launches
    achieved = launch_bytes / launch_s / 1e9
    if kernel != "regdecode":
        layer_traffic = None  # the capture was of the register-decode kernel
    traffic = None if layer_traffic is None else round(layer_traffic * layers / stack.launches)
    roofline = {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "traffic": traffic,
                "peak_source": peak_kind + " (MEASURED_PEAKS.json hbm_gbs, copy burst)",
                "kernel": {"regdecode": "gemv_kernel<1>", "tcgen05": "tc_gemv_kernel",
                           "mma": "mma_gemm_kernel"}[kernel] +
                          " (aq_decode_step_weights: one launch per projection)",
                "algorithmic_bytes_per_launch": round(launch_bytes)}

    cpu = None
    if dist.rank == 0 and not a.no_extras:
        cpu = cpu_baseline(shapes, a.m)

    clocks = sampler.summary() if sampler else None
    out = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s",
        "n_gpus": dist.world, "steps": a.steps, "warmup": a.warmup,
        "ms_per_step": round(ms, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "nvfp4 weights, bf16 activations, fp32 accumulate",
        "data": "synthetic (seeded N(0,0.02^2) weights with 0.1% x20 outliers, N(0,1) tokens)",
        "pct_of_8tbs": round(100.0 * value / dist.world / NOMINAL_HBM_GBS, 2),
        "config": {"workload": name, "layers": layers,
                   "projections": [list(s) for s in shapes], "m": a.m,
                   "weight_bytes_per_step": weight_bytes(shapes, layers),
                   "algorithmic_bytes_per_step": step_bytes,
                   "launch": "aq_decode_step_weights (PDL) captured in one CUDA graph, "
                             "%d GEMV launches per step" % stack.launches,
                   "l2": "inputs larger than L2 (weights %.1f GB per step)" %
                         (weight_bytes(shapes, layers) / 1e9),
                   "parallelism": "replicas x%d" % dist.world},
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": a.steps * stack.launches,
        "clocks": clocks,
        "extras": extras,
    }
    if dist.rank == 0:
        print(json.dumps(out), flush=True)


# ------------------------------------------------------------ batch sweep

SWEEP_M = (1, 2, 4, 8, 16, 32, 64)


def run_bf16_lm_head(a, dist):
    """One JSON line for the bf16 GEMV leg alone (its own configuration, not
    the headline)."""
    import torch
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(dist.local)
    device = torch.device("cuda", dist.local)
    stream = torch.cuda.Stream(device)
    r = bf16_lm_head_leg(stream, dist, a, device)
    if dist.rank == 0:
        print(json.dumps({"metric": "bf16 GEMV HBM GB/s", "value": r["GBps"], "unit": "GB/s",
                          "n_gpus": dist.world, "higher_is_better": True,
                          "data": "synthetic (seeded N(0,0.02^2) weight, N(0,1) token)",
                          "config": {"workload": "~31B tied lm_head, bf16", **r}}), flush=True)


def run_load_time(a, dist):
    """The load-time kernels of the path: theta bundle -> W_eff -> NVFP4
    (aq_reconstruct_quantize_nvfp4, rank 4) and NVFP4 of a bf16 weight
    (aq_quantize_nvfp4), on the 1B-shaped MLP weights (fused gate+up
    [13824, 1152], down [1152, 6912]) and the ~31B fused gate+up [43008,
    5376].  Each call rotates over enough input copies to exceed L2 twice
    and is event-timed on the launching stream.  Algorithmic bytes: 2 B read
    + 0.5625 B written per element + 4 B of g_dec, plus the theta (4 n +
    2 (n + k) r bytes) for the fused form."""
    import torch
    from nvfp4_block_scaled_aq_gb300 import aq, inputs
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(dist.local)
    device = torch.device("cuda", dist.local)
    stream = torch.cuda.Stream(device)
    r = 4
    shapes = [("1b_gate_up", 13824, 1152), ("1b_down", 1152, 6912), ("31b_gate_up", 43008, 5376)]
    qws = torch.zeros(aq.quantize_workspace_bytes(), dtype=torch.uint8, device=device)
    rows = []
    for name, n, k in shapes:
        copies = max(1, -(-(256 << 20) // (2 * n * k)))
        thetas = [inputs.theta(n, k, r, seed=inputs.seed_of(9500 + i), device=device)
                  for i in range(copies)]
        out = aq.Nvfp4Weight.empty(n, k, device=device)
        torch.cuda.synchronize()
        res = {"shape": [n, k], "rank": r, "copies": copies}
        for form in ("reconstruct_quantize", "quantize"):
            def call(i):
                th = thetas[i % copies]
                if form == "quantize":
                    aq.quantize(th.W0, out, qws, stream=stream)
                else:
                    aq.reconstruct_quantize(th.W0, th.s, th.U, th.V, out, qws, stream=stream)
            reps = max(2 * copies, 10)
            with torch.cuda.stream(stream):
                for i in range(max(a.warmup, copies)):
                    call(i)
                stream.synchronize()
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                for i in range(reps):
                    call(i)
                e1.record(stream)
            torch.cuda.synchronize()
            secs = e0.elapsed_time(e1) / 1e3 / reps
            byts = load_time_bytes(n, k, r, form == "reconstruct_quantize")
            res[form] = {"us_per_call": round(secs * 1e6, 2), "GBps": round(byts / secs / 1e9, 1),
                         "algorithmic_bytes": byts}
        st = aq.poll_device_status()
        if st != aq.OK:
            raise RuntimeError("load-time kernels reported %s: %s" % (st, aq.last_error()))
        rows.append(dict(name=name, **res))
        del thetas
    peak, src = load_peaks()
    if dist.rank == 0:
        # the headline: the fused call on the largest shape (the ~31B gate+up)
        head = max(rows, key=lambda row: row["shape"][0] * row["shape"][1])
        print(json.dumps({"metric": "load-time reconstruct + NVFP4 quantise, GB/s of algorithmic bytes",
                          "value": head["reconstruct_quantize"]["GBps"], "unit": "GB/s",
                          "n_gpus": dist.world, "higher_is_better": True,
                          "data": "synthetic (seeded theta bundles, N(0, 0.02^2) W0)",
                          "config": {"workload": "load-time kernels on the 1B MLP and ~31B gate+up shapes",
                                     "value_of": "%s fused reconstruct + quantise" % head["name"],
                                     "l2": "inputs rotated over copies exceeding 256 MB"},
                          "hbm_peak_gbs": peak, "hbm_peak_source": src, "shapes": rows}), flush=True)


def run_sweep(a, dist):
    """GEMV kernels vs the block-scaled MMA path on the ~31B-shaped fused
    gate+up [43008, 5376] and down [5376, 21504] weights.  Each timing is a
    CUDA graph of back-to-back calls that rotate over enough weight copies
    to exceed L2, replayed between CUDA events on the launching stream."""
    import torch
    from nvfp4_block_scaled_aq_gb300 import aq, inputs
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(dist.local)
    device = torch.device("cuda", dist.local)
    stream = torch.cuda.Stream(device)
    qws = torch.zeros(aq.quantize_workspace_bytes(), dtype=torch.uint8, device=device)
    results = []
    ms = tuple(int(v) for v in a.sweep_m.split(",")) if a.sweep_m else SWEEP_M
    projs = {"both": (2, 3), "gate_up": (2,), "down": (3,)}[a.sweep_proj]
    for proj in projs:
        n, k = inputs.LAYER_31B[proj]
        wbytes = n * k // 2 + n * k // 16
        copies = max(2, -(-3 * 129 * 2 ** 20 // wbytes))  # at least ~3x L2 in rotation
        weights = []
        for c in range(copies):
            W = inputs.weight(n, k, seed=inputs.seed_of(0, c, proj), device=device)
            w = aq.Nvfp4Weight.empty(n, k, device=device)
            aq.quantize(W, w, qws)
            del W
            weights.append(w)
        torch.cuda.synchronize()  # everything below runs on `stream`
        for m in ms:
            x = inputs.tokens(m, k, seed=inputs.seed_of(1, 0, proj) + m, device=device)
            y = torch.empty((m, n), dtype=torch.bfloat16, device=device)
            ws = torch.zeros(aq.gemv_workspace_bytes(n, k, m), dtype=torch.uint8, device=device)
            torch.cuda.synchronize()  # x, y and ws are ready before `stream` uses them
            paths = [("mma", aq.PATH_MMA)]
            if m <= aq.MAX_M:
                paths.insert(0, ("gemv_regdecode", aq.PATH_GEMV_REGDECODE))
            if m <= 5:
                paths.insert(1, ("gemv_tcgen05", aq.PATH_GEMV_TCGEN05))
            row = {"proj": "gate_up" if proj == 2 else "down", "n": n, "k": k, "m": m}
            alg = wbytes + 4 + 2 * m * k + 2 * m * n
            for name, path in paths:
                calls = 4 * copies
                g = torch.cuda.CUDAGraph()
                with torch.cuda.stream(stream):
                    for w in weights:
                        aq.gemv(w, x, y, ws, path=path, stream=stream)
                    stream.synchronize()
                    with torch.cuda.graph(g, stream=stream):
                        for i in range(calls):
                            aq.gemv(weights[i % copies], x, y, ws, path=path, stream=stream)

                def run():
                    with torch.cuda.stream(stream):
                        g.replay()
                reps = max(3, a.steps // 20)
                secs = time_region(run, reps, max(3, a.warmup), stream, dist)
                us = secs / (reps * calls) * 1e6
                row[name] = {"us": round(us, 2), "GBps": round(alg / us / 1e3, 1)}
                del g
            st = aq.poll_device_status()
            if st != aq.OK:
                raise RuntimeError("device status %d in the sweep" % st)
            results.append(row)
            torch.cuda.synchronize()  # `stream` is done with x, y and ws before they are freed
        torch.cuda.synchronize()
        del weights
    crossover = {}
    for pname in ("gate_up", "down"):
        rows = [r for r in results if r["proj"] == pname]
        cross = None
        for r in rows:
            gemv = [r[kname]["us"] for kname in ("gemv_regdecode", "gemv_tcgen05") if kname in r]
            if gemv and r["mma"]["us"] < min(gemv):
                cross = r["m"]
                break
        crossover[pname] = cross
    peak, peak_kind = load_peaks()
    out = {"metric": "NVFP4 GEMV vs block-scaled MMA, us per call and GB/s by batch",
           "value": None, "unit": "GB/s", "n_gpus": dist.world,
           "higher_is_better": True, "data": "synthetic (seeded)",
           "config": {"workload": "batch sweep on ~31B-shaped fused gate+up [43008, 5376] and "
                                  "down [5376, 21504]", "m": list(ms),
                      "l2": "each graph rotates over enough weight copies to exceed L2"},
           "sweep": results,
           "crossover_m_mma_faster": crossover,
           "hbm_peak_gbs": peak, "hbm_peak_source": peak_kind}
    if dist.rank == 0:
        print(json.dumps(out), flush=True)


# ------------------------------------------------------------ reference arm

def run_reference(a, dist):
    """The CPU oracle as it stands, on every host core, on a bounded sample
    of the same workload: each step is the oracle's GEMV over 64 rows per
    host core of each of layer 0's projections, one thread per core (ctypes
    releases the GIL for the C call)."""
    if dist.rank != 0:
        return
    import concurrent.futures as cf
    import numpy as np
    import oracle
    name, shapes, layers = workload(a.workload)
    m = a.m
    model, cores = host_cpu()
    prepared = oracle_rows(shapes, m, max_rows=64 * cores)
    step_bytes = sum(r * (k // 2 + k // 16) + 2 * m * k + 2 * m * r + 4
                     for _, _, _, _, r, k in prepared)
    jobs = [(packed, scales, gd, x, np.arange(r0, min(rows, r0 + 64)))
            for packed, scales, gd, x, rows, k in prepared for r0 in range(0, rows, 64)]
    ex = cf.ThreadPoolExecutor(max_workers=cores)

    def step():
        list(ex.map(lambda j: oracle.gemv(j[0], j[1], j[2], j[3], rows=j[4]), jobs))
    for _ in range(a.warmup):
        step()
    t = time.perf_counter()
    for _ in range(a.steps):
        step()
    secs = time.perf_counter() - t
    ex.shutdown()
    value = step_bytes * a.steps / secs / 1e9
    sample = ("%d rows of each of layer 0's 4 projections per step (%d of %d weight bytes "
              "of a full step), m=%d, fp64 accumulation, %d threads" %
              (64 * cores, sum(r * (k // 2 + k // 16) for _, _, _, _, r, k in prepared),
               weight_bytes(shapes, layers), m, cores))
    out = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
           "n_gpus": dist.world, "steps": a.steps, "warmup": a.warmup,
           "ms_per_step": round(secs / a.steps * 1e3, 3), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64 accumulate (CPU oracle)",
           "data": "synthetic (seeded, drawn on the CPU)",
           "config": {"workload": name + " (bounded sample)", "m": m},
           "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores,
                            "kind": "oracle", "cpu": model, "sample": sample},
           "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def main():
    a = parse()
    dist = Dist()
    try:
        if a.impl == "reference":
            run_reference(a, dist)
        elif a.batch_sweep:
            run_sweep(a, dist)
        elif a.bf16_lm_head:
            run_bf16_lm_head(a, dist)
        elif a.load_time:
            run_load_time(a, dist)
        elif a.small_configs:
            run_small_configs(a, dist)
        elif a.profile_case:
            run_profile_case(a, dist)
        else:
            run_aq(a, dist)
    finally:
        dist.close()


if __name__ == "__main__":
    main()
