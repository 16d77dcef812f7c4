"""Benchmark of the Flint MoE FFN layer on B300.

Headline workload: the decode stack -- 47 distinct BF16 MoE layers of the
H=2048 / I=512 / 256+1-expert shape (about 76 GB of weights resident, far
larger than L2), per-expert router bias ~ N(0, 0.5), T=1 token per layer
step, the layers applied one after another to the same x.  One step is one
pass over the 47 layers (replayed as one CUDA graph).  Metric: MoE-layer
tokens per second = 47 * T / step time, and us per layer; roofline: unique
bytes of touched expert weights per layer / us per layer, against the
measured HBM copy bandwidth (and, beside it, the 8 TB/s nominal peak).

The default run (--workload all) then times, in the same process, the
other configurations of the metric and reports each under "configs": the
BF16 stack at T=8 and T=32 (clustered tokens), the T=8192 prefill on the
stack's first layer (tensor-core roofline) and the NVFP4 (W4A16) stack at
T=1, 8 and 32.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl flint|reference]
                    [--workload all|decode1|decode8|decode32|prefill8192|
                                nvfp4_decode1|nvfp4_decode8|nvfp4_decode32]

--impl reference times the fp64 CPU oracle on the host cores (a bounded
sample of the headline workload per step).  With N > 1 each rank runs its own
replica of the stack (the layer does not shard; no collective on the data
path); value is the sum over ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

N_LAYERS = 47
EXPERT_BYTES_BF16 = 3 * 2048 * 512 * 2        # 6,291,456
ROUTER_BYTES = 256 * 2048 * 2 + 256 * 4
WORKLOADS = {
    "decode1": {"T": 1, "x": "gauss", "x_seed": 11},
    "decode8": {"T": 8, "x": "clustered", "x_seed": 12},
    "decode32": {"T": 32, "x": "clustered", "x_seed": 13},
    "prefill8192": {"T": 8192, "x": "gauss", "x_seed": 14, "prefill": True},
    "nvfp4_decode1": {"T": 1, "x": "gauss", "x_seed": 11, "nvfp4": True},
    "nvfp4_decode8": {"T": 8, "x": "clustered", "x_seed": 12, "nvfp4": True},
    "nvfp4_decode32": {"T": 32, "x": "clustered", "x_seed": 13, "nvfp4": True},
    "nvfp4_prefill8192": {"T": 8192, "x": "gauss", "x_seed": 14, "prefill": True, "nvfp4": True},
    "nvfp4_lm_head1": {"T": 1, "x": "gauss", "x_seed": 11, "lm_head": True},
    "nvfp4_lm_head32": {"T": 32, "x": "clustered", "x_seed": 13, "lm_head": True},
}
LM_HEAD_V = 131072        # assumed vocabulary (not on the pages): the head is about 10.7% of 2.5B active
LM_HEAD_SEED = 5
LM_HEAD_SAMPLE_ROWS = 2048   # rows of the head the oracle evaluates per CPU-baseline step
# dense flops of one layer per token: 7 experts x (gate, up, down) + router
FLOPS_PER_TOKEN = 7 * 2 * 3 * 2048 * 512 + 2 * 256 * 2048
GATE_UP_BYTES = 2 * 512 * 2048 * 2            # one expert's gate and up matrices, bf16
DOWN_BYTES = 2048 * 512 * 2                   # one expert's down matrix, bf16
# NVFP4: E2M1 codes (half a byte per weight) + one E4M3 scale per 16 weights + an fp32 scale per matrix
NV_GATE_UP_BYTES = 2 * 512 * 2048 // 2 + 2 * 512 * 2048 // 16 + 4     # 1,179,652
NV_DOWN_BYTES = 2048 * 512 // 2 + 2048 * 512 // 16 + 4                  # 589,828
STACK_MAX_T = 8                               # FLINT_STACK_MAX_T: the persistent stack kernel's batch limit
# kernel ids of flint_moe_set_kernel_events (include/flint_moe.h)
K_ROUTER, K_GATE_UP, K_DOWN, K_COMBINE = 0, 1, 2, 3
# the source files each timed kernel is built from (for the ncu traffic record)
KERNEL_SOURCES = {
    "gateup_nvfp4_kernel": ["decode_nvfp4.cu", "mma_sync.cuh", "routing.cuh", "flint_common.cuh"],
    "gateup_mma_kernel": ["decode_mma.cu", "mma_sync.cuh", "routing.cuh", "flint_common.cuh"],
    "down_mma_kernel": ["decode_mma.cu", "mma_sync.cuh", "routing.cuh", "flint_common.cuh"],
    "down_nvfp4_kernel": ["decode_nvfp4.cu", "mma_sync.cuh", "routing.cuh", "flint_common.cuh"],
    "prefill_gateup_kernel": ["prefill.cu", "prefill_common.cuh", "tc_ptx.cuh", "flint_common.cuh"],
    "prefill_down_kernel": ["prefill.cu", "prefill_common.cuh", "tc_ptx.cuh", "flint_common.cuh"],
    "prefill_gateup_nvfp4_kernel": ["prefill_nvfp4.cu", "prefill_common.cuh", "tc_ptx.cuh",
                                    "flint_common.cuh"],
    "prefill_down_nvfp4_kernel": ["prefill_nvfp4.cu", "prefill_common.cuh", "tc_ptx.cuh",
                                  "flint_common.cuh"],
    "lm_head_nvfp4_kernel": ["lm_head.cu", "mma_sync.cuh", "nvfp4_frag.cuh", "flint_common.cuh"],
    "stack_decode_kernel": ["stack_decode.cu", "mma_sync.cuh", "nvfp4_frag.cuh", "routing.cuh", "flint_common.cuh"],
}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="flint", choices=["flint", "reference"])
    ap.add_argument("--workload", default="all", choices=["all"] + sorted(WORKLOADS))
    ap.add_argument("--layers", type=int, default=N_LAYERS, help=argparse.SUPPRESS)
    return ap.parse_args()


def peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))), "measured"
    except Exception:
        return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}, "fallback"


# NVML clock-event reason bits (nvml.h: nvmlClocksEventReason*)
_REASON_BITS = {"nvmlClocksEventReasonSwPowerCap": 0x4, "nvmlClocksEventReasonHwSlowdown": 0x8,
                "nvmlClocksEventReasonSwThermalSlowdown": 0x20, "nvmlClocksEventReasonHwThermalSlowdown": 0x40,
                "nvmlClocksEventReasonHwPowerBrakeSlowdown": 0x80}


class _CtypesNvml:
    """The few read-only NVML queries the sampler needs, through libnvidia-ml."""
    NVML_CLOCK_SM = 1

    def __init__(self):
        import ctypes
        self.c = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")

    def nvmlInit(self):
        if self.lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")

    def nvmlDeviceGetHandleByPciBusId(self, bus):
        h = self.c.c_void_p()
        if self.lib.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), self.c.byref(h)) != 0:
            raise RuntimeError("nvmlDeviceGetHandleByPciBusId failed")
        return h

    def _clock(self, fn, h, kind):
        v = self.c.c_uint()
        if fn(h, kind, self.c.byref(v)) != 0:
            raise RuntimeError("nvml clock query failed")
        return v.value

    def nvmlDeviceGetClockInfo(self, h, kind):
        return self._clock(self.lib.nvmlDeviceGetClockInfo, h, kind)

    def nvmlDeviceGetMaxClockInfo(self, h, kind):
        return self._clock(self.lib.nvmlDeviceGetMaxClockInfo, h, kind)

    def nvmlDeviceGetCurrentClocksEventReasons(self, h):
        v = self.c.c_ulonglong()
        fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons
        if fn(h, self.c.byref(v)) != 0:
            raise RuntimeError("nvml reasons query failed")
        return v.value


class ClockSampler:
    """SM clock and clock-event reasons sampled by NVML every ~2 ms while the
    timed region runs (read-only queries; nothing is changed on the GPU)."""

    REASONS = [("hw_slowdown", "nvmlClocksEventReasonHwSlowdown"),
               ("hw_thermal_slowdown", "nvmlClocksEventReasonHwThermalSlowdown"),
               ("sw_thermal_slowdown", "nvmlClocksEventReasonSwThermalSlowdown"),
               ("sw_power_cap", "nvmlClocksEventReasonSwPowerCap"),
               ("hw_power_brake", "nvmlClocksEventReasonHwPowerBrakeSlowdown")]

    def __init__(self, torch_device):
        import threading
        self.dev = torch_device
        self.samples = []
        self.stop = threading.Event()
        self.thread = None
        self.err = None

    def _handle(self):
        import torch
        pr = torch.cuda.get_device_properties(self.dev)
        bus = f"{pr.pci_domain_id:08x}:{pr.pci_bus_id:02x}:{pr.pci_device_id:02x}.0"
        try:
            import pynvml
        except ImportError:
            pynvml = _CtypesNvml()
        pynvml.nvmlInit()
        return pynvml, pynvml.nvmlDeviceGetHandleByPciBusId(bus)

    def _run(self):
        try:
            nv, h = self._handle()
            mx = nv.nvmlDeviceGetMaxClockInfo(h, nv.NVML_CLOCK_SM)
            while not self.stop.is_set():
                sm = nv.nvmlDeviceGetClockInfo(h, nv.NVML_CLOCK_SM)
                rs = nv.nvmlDeviceGetCurrentClocksEventReasons(h)
                self.samples.append((sm, mx, rs))
                self.stop.wait(0.002)
        except Exception as e:  # NVML missing: report unsampled
            self.err = repr(e)

    def __enter__(self):
        import threading
        self.thread = threading.Thread(target=self._run, daemon=True)
        self.thread.start()
        import time as _t
        _t.sleep(0.05)
        return self

    def __exit__(self, *a):
        self.stop.set()
        if self.thread:
            self.thread.join(timeout=5)

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0,
                    "error": self.err}
        reasons = set()
        for _, _, rs in self.samples:
            for name, const in self.REASONS:
                if rs & _REASON_BITS[const]:
                    reasons.add(name)
        return {"sm_mhz": statistics.median(s[0] for s in self.samples),
                "sm_max_mhz": max(s[1] for s in self.samples), "reasons": sorted(reasons),
                "samples": len(self.samples), "source": "nvml"}


def dist_setup(args):
    import torch
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if args.impl == "flint" else "gloo"
        if args.impl == "flint":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return ws, rank, local


def max_over_ranks(values, device="cuda"):
    """Element-wise maximum of this rank's timings over all ranks (the
    slowest rank sets the job's time); the values themselves at N = 1."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def whole_job_rate(units_per_rank, ws, ms):
    """Units per second of the whole job: every rank processed units_per_rank
    in at most ms milliseconds."""
    return ws * units_per_rank / (ms * 1e-3)


def sources_digest(kernel):
    """sha1 of the sources `kernel` is compiled from."""
    import hashlib
    h = hashlib.sha1()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "sparse_moe_transformer_03_b300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def traffic_from_profiles(kernel, workload):
    """DRAM bytes (read + write) per launch of `kernel` on `workload` from
    the ncu record in profiles/dram_traffic.md, or None when there is none or
    the kernel's sources changed since it was taken."""
    try:
        lines = open(os.path.join(ROOT, "profiles", "dram_traffic.md")).read().splitlines()
    except OSError:
        return None
    digest = sources_digest(kernel)
    for ln in lines:
        f = [c.strip() for c in ln.strip().strip("|").split("|")]
        if len(f) >= 4 and f[0] == kernel and f[1] == workload and f[3] == digest:
            try:
                return float(f[2])
            except ValueError:
                return None
    return None


def kernel_durations(flint, torch, stream, calls, kid, nsteps):
    """Device durations (ms) of kernel `kid` in every forward of `calls`
    (a list of (handle, x, T, y)), over nsteps passes launched directly: the
    library records a CUDA event pair on `stream` immediately around that
    kernel's launch (flint_moe_set_kernel_events)."""
    evs = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in calls]
           for _ in range(nsteps)]
    with torch.cuda.stream(stream):
        for st in range(nsteps):
            for (h, x, T, y), (e0, e1) in zip(calls, evs[st]):
                flint.flint_moe_set_kernel_events(h, kid, e0, e1)
                flint.flint_moe_forward(h, x, T, y, stream)
    stream.synchronize()
    for (h, _, _, _) in calls:
        flint.flint_moe_set_kernel_events(h, -1)
    return [[e0.elapsed_time(e1) for (e0, e1) in row] for row in evs]


def x_bits_for(wl):
    from synth import gen
    if wl["x"] == "gauss":
        return gen.x_gaussian(wl["x_seed"], wl["T"])
    return gen.x_clustered(wl["x_seed"], wl["T"])[0]


# ---------------------------------------------------------------------------
# reference arm: the fp64 oracle on the host cores
# ---------------------------------------------------------------------------

def run_reference(args, wl, ws, rank):
    """The oracle as it stands on the host cores: each step a bounded sample
    of the workload (two layers of the decode stack, or the first
    PREFILL_SAMPLE tokens of the prefill input on its one layer)."""
    from synth import device

    if rank != 0:
        return
    device.build()
    T = wl["T"]
    xb = x_bits_for(wl)
    if wl.get("lm_head"):
        run_reference_lm_head(args, wl, xb)
        return
    prefill = bool(wl.get("prefill"))
    n_layers = 1 if prefill else 2
    xs = xb[:PREFILL_SAMPLE] if prefill else xb
    orcs = []
    for l in range(n_layers):
        lw = device.LayerWeights(1, l, True)
        orc = layer_oracle(lw, device.LayerNVFP4(lw) if wl.get("nvfp4") else None)
        orc.forward(xs)    # copies the touched experts to the host (untimed)
        orcs.append(orc)
        del lw
    cores = os.cpu_count() or 1
    times = []
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        for orc in orcs:
            orc.forward(xs)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            times.append(dt)
    step = sum(times) / len(times)
    if prefill:
        value, unit = len(xs) / step, "tokens/s"
        metric = f"MoE-layer tokens/s, prefill T={T}"
        workload = (f"prefill: one BF16 MoE layer (H=2048, I=512, 256 routed + 1 shared, top-6 sigmoid, router bias "
                    f"N(0,0.5)), T={T} tokens (x ~ N(0,1) RMS-normalised, seed {wl['x_seed']}); "
                    f"sample of the first {len(xs)} tokens per step")
        sample = f"first {len(xs)} of the {T} prefill tokens, one layer, touched experts on the host"
        us_layer = step * 1e6 * T / len(xs)
    else:
        value, unit = n_layers * T / step, "layer-tokens/s"
        kind = "NVFP4" if wl.get("nvfp4") else "BF16"
        metric = f"MoE-layer tokens/s, {'NVFP4 ' if wl.get('nvfp4') else ''}decode stack T={T}"
        workload = f"decode stack, {N_LAYERS} {kind} MoE layers, T={T}, sample of {n_layers} layers per step"
        sample = f"{n_layers} layers of the stack at T={T}, touched experts on the host"
        us_layer = step * 1e6 / n_layers
    line = {"metric": metric, "value": value, "unit": unit,
            "impl": "reference", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": step * 1e3, "higher_is_better": True, "scaling": "weak",
            "us_per_layer": us_layer, "dtype": "f64", "data": "synthetic",
            "config": {"workload": workload, "H": 2048, "I": 512, "experts": 257, "top_k": 6},
            "vs_baseline": None,
            "cpu_baseline": {"value": value, "unit": unit, "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_reference_lm_head(args, wl, xb):
    """The oracle on the first LM_HEAD_SAMPLE_ROWS rows of the output layer
    per step (the head generated and quantised by the input generator, not
    by the library), scaled to the whole vocabulary."""
    import torch
    import oracle
    from synth import device, gen
    # the tensor scale depends on the whole head: quantise all of it, keep the sample rows
    full = torch.empty((LM_HEAD_V, gen.H), dtype=torch.bfloat16, device="cuda")
    device.fill_normal_bf16(full, LM_HEAD_SEED, 0, gen.T_LM_HEAD, gen.WEIGHT_STD)
    pk, sc, ts = device.nvfp4_quantize(full)
    m = oracle.Mat(packed=pk[0][:LM_HEAD_SAMPLE_ROWS].cpu().numpy(), scales=sc[0][:LM_HEAD_SAMPLE_ROWS].cpu().numpy(),
                   tensor_scale=float(ts[0].item()))
    del full, pk, sc
    times = []
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        oracle.lm_head(xb, m)
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    step = sum(times) / len(times) * LM_HEAD_V / LM_HEAD_SAMPLE_ROWS
    T = wl["T"]
    value, unit = T / step, "tokens/s"
    sample = (f"first {LM_HEAD_SAMPLE_ROWS} of the {LM_HEAD_V} head rows at T={T} per step, scaled by "
              f"{LM_HEAD_V // LM_HEAD_SAMPLE_ROWS} to the whole head")
    line = {"metric": f"output-layer tokens/s, NVFP4 lm_head T={T}", "value": value, "unit": unit,
            "impl": "reference", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": step * 1e3, "higher_is_better": True, "scaling": "weak", "us_per_call": step * 1e6,
            "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"output layer: NVFP4 head [{LM_HEAD_V}][2048], T={T}; {sample}"},
            "vs_baseline": None,
            "cpu_baseline": {"value": value, "unit": unit, "cores": 1, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# flint arm
# ---------------------------------------------------------------------------

def layer_oracle(lw, q=None):
    """The oracle of a device layer: bf16 experts, or the NVFP4 encoding q of them."""
    import oracle
    from oracle.reference import LayerOracle
    if q is None:
        return LayerOracle.from_bf16_layer(lw)

    def mats(e):
        (pg, sg, tg), (pd, sd, td) = q.expert_parts(e)
        return (oracle.Mat(packed=pg, scales=sg, tensor_scale=tg),
                oracle.Mat(packed=pd, scales=sd, tensor_scale=td))
    return LayerOracle(lw.router_bits(), lw.bias_host(), mats, mats(lw.E), lw.E)


def cpu_baseline(wl, stack_layers, seconds=10.0):
    """The oracle, as it stands, on one decode step of a 2-layer sample
    (stack_layers: bf16 layers, or (bf16 layer, NVFP4 encoding) pairs), for
    about `seconds` of host time."""
    T = wl["T"]
    xb = x_bits_for(wl)
    n = 2
    orcs = [layer_oracle(*(stack_layers[l] if isinstance(stack_layers[l], tuple) else (stack_layers[l],)))
            for l in range(n)]
    for o in orcs:
        o.forward(xb)                  # host copies of touched experts (untimed)
    t0 = time.perf_counter()
    reps = 0
    while True:
        for o in orcs:
            o.forward(xb)
        reps += 1
        if time.perf_counter() - t0 > seconds or reps >= 50:
            break
    dt = (time.perf_counter() - t0) / reps
    return {"value": n * T / dt, "unit": "layer-tokens/s", "cores": os.cpu_count() or 1, "kind": "oracle",
            "sample": f"{n} layers of the decode stack at T={T} (touched experts copied to host, copy untimed), {reps} reps"}


PREFILL_SAMPLE = 256   # tokens of the prefill input the oracle runs per step


def cpu_baseline_prefill(wl, lw, xb, seconds=10.0, q=None):
    """The oracle, as it stands, on the first PREFILL_SAMPLE tokens of the prefill input
    (bf16 experts, or their NVFP4 encoding q)."""
    orc = layer_oracle(lw, q)
    xs = xb[:PREFILL_SAMPLE]
    orc.forward(xs)                    # host copies of touched experts (untimed)
    t0 = time.perf_counter()
    reps = 0
    while True:
        orc.forward(xs)
        reps += 1
        if time.perf_counter() - t0 > seconds or reps >= 20:
            break
    dt = (time.perf_counter() - t0) / reps
    return {"value": PREFILL_SAMPLE / dt, "unit": "tokens/s", "cores": os.cpu_count() or 1, "kind": "oracle",
            "sample": f"first {PREFILL_SAMPLE} of the {wl['T']} prefill tokens, one layer "
                      f"(touched experts copied to host, copy untimed), {reps} reps"}


def timed_ms(torch, stream, fn, n):
    """Mean device time (ms) of n calls of fn, CUDA events on `stream`."""
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    ev[0].record(stream)
    for _ in range(n):
        fn()
    ev[1].record(stream)
    ev[1].synchronize()
    return ev[0].elapsed_time(ev[1]) / n


def hbm_roof(achieved_gbs, peak_gbs, pk_kind):
    """An HBM roofline entry: the fraction of the measured copy bandwidth and,
    beside it, the fraction of the 8 TB/s nominal HBM3e peak."""
    return {"achieved": achieved_gbs, "peak": peak_gbs, "unit": "GB/s", "frac": achieved_gbs / peak_gbs,
            "peak_kind": f"{pk_kind} HBM copy bandwidth (burst)",
            "frac_vs_8tbs": achieved_gbs / NOMINAL_HBM_GBS}


NOMINAL_HBM_GBS = 8000.0


def build_bf16_stack(flint, device, L, keep=2):
    """L distinct BF16 layers of the decode stack (seed 1, skewed router bias).
    The handle copies the experts into its own tiled layout, so the generated
    bf16 experts are dropped after create except for the first `keep` layers
    (the oracle samples them); the routers stay (the handle borrows them)."""
    import torch
    layers, handles = [], []
    for l in range(L):
        lw = device.LayerWeights(1, l, True)
        handles.append(flint.flint_moe_create(lw.router_W, lw.router_b, list(lw.gate_up[:256]), list(lw.down[:256]),
                                              (lw.gate_up[256], lw.down[256])))
        if l >= keep:
            lw.gate_up = lw.down = None
        layers.append(lw)
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return layers, handles


def build_nvfp4_stack(flint, device, L, keep=2):
    """The same stack with NVFP4-encoded experts; the handle repacks them into
    memory it owns, so only the first `keep` layers' encodings (for the oracle)
    and every layer's router are kept."""
    import torch
    layers, handles = [], []
    for l in range(L):
        lw = device.LayerWeights(1, l, True)
        q = device.LayerNVFP4(lw)
        gu, dn, sh = q.create_args()
        handles.append(flint.flint_moe_create(lw.router_W, lw.router_b, gu, dn, sh, dtype=flint.FLINT_NVFP4))
        lw.gate_up = lw.down = None
        layers.append((lw, q) if l < keep else (lw, None))
        del gu, dn, sh
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return layers, handles


def bench_decode(args, wl, name, layers, handles, ws, rank, nv, cpu_seconds):
    """One decode configuration on a built stack: the L forwards of a step
    replayed as one CUDA graph (weights far larger than L2, so each step
    reads them from HBM again), plus the per-kernel rooflines, e2e through the
    C ABI and the oracle's CPU baseline."""
    import numpy as np
    import torch
    from sparse_moe_transformer_03_b300 import flint

    T = wl["T"]
    L = len(handles)
    pk, pk_kind = peaks()
    xb = x_bits_for(wl)
    x = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).cuda()
    y_all = torch.empty((L, T, 2048), dtype=torch.bfloat16, device="cuda")
    ys = [y_all[l] for l in range(L)]
    # T <= 8: the whole stack in one persistent launch (flint_moe_forward_layers)
    use_stack = T <= STACK_MAX_T

    # unique touched experts per layer (for the algorithmic byte count)
    uniq = []
    for h in handles:
        idx = torch.empty((T, 6), dtype=torch.int32, device="cuda")
        w = torch.empty((T, 6), dtype=torch.float32, device="cuda")
        flint.flint_moe_route_only(h, x, None, T, idx, w)
        uniq.append(len(set(idx.cpu().numpy().ravel().tolist())))
    per_expert = NV_GATE_UP_BYTES + NV_DOWN_BYTES if nv else EXPERT_BYTES_BF16
    bytes_per_step = sum((u + 1) * per_expert for u in uniq)

    stream = torch.cuda.Stream()
    torch.cuda.synchronize()

    def step_direct():
        for l in range(L):
            flint.flint_moe_forward(handles[l], x, T, ys[l], stream)

    with torch.cuda.stream(stream):
        step_direct()
        step_direct()
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step_direct()
    stream.synchronize()

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            graph.replay()
    stream.synchronize()
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(torch.cuda.current_device()) as clk:
        with torch.cuda.stream(stream):
            ms = timed_ms(torch, stream, graph.replay, args.steps)
    torch.cuda.synchronize()
    clocks = clk.summary()
    with torch.cuda.stream(stream):
        ms_direct = timed_ms(torch, stream, step_direct, max(3, args.steps // 2))

    # end to end through the C ABI: pinned host x -> device, the stack, every y -> host
    x_host = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).pin_memory()
    y_host = torch.empty((L, T, 2048), dtype=torch.bfloat16).pin_memory()
    x_dev = torch.empty_like(x)

    def step_e2e():
        x_dev.copy_(x_host, non_blocking=True)
        if use_stack:
            flint.flint_moe_forward_layers(handles, [x_dev] * L, T, ys, stream)
        else:
            for l in range(L):
                flint.flint_moe_forward(handles[l], x_dev, T, ys[l], stream)
        y_host.copy_(y_all, non_blocking=True)

    with torch.cuda.stream(stream):
        for _ in range(3):
            step_e2e()
        ms_e2e = min(timed_ms(torch, stream, step_e2e, max(3, args.steps // 2)) for _ in range(3))
    stream.synchronize()

    ms_layers = ms
    stack = None
    if use_stack:
        def step_stack():
            flint.flint_moe_forward_layers(handles, [x] * L, T, ys, stream)
        with torch.cuda.stream(stream):
            step_stack()
        stream.synchronize()
        sgraph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(sgraph, stream=stream):
            step_stack()
        with torch.cuda.stream(stream):
            for _ in range(args.warmup):
                sgraph.replay()
        stream.synchronize()
        if ws > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        with ClockSampler(torch.cuda.current_device()) as clk_s:
            with torch.cuda.stream(stream):
                ms_stack = timed_ms(torch, stream, sgraph.replay, args.steps)
        torch.cuda.synchronize()
        clocks = clk_s.summary()
        with torch.cuda.stream(stream):
            ms_direct = timed_ms(torch, stream, step_stack, max(3, args.steps // 2))
        # the persistent kernel alone: events around its launch (one per step)
        ksteps = max(3, min(args.steps, 10))
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(ksteps)]
        with torch.cuda.stream(stream):
            for e0, e1 in evs:
                flint.flint_moe_set_kernel_events(handles[0], K_GATE_UP, e0, e1)
                flint.flint_moe_forward_layers(handles, [x] * L, T, ys, stream)
        stream.synchronize()
        flint.flint_moe_set_kernel_events(handles[0], -1)
        k_ms = sum(e0.elapsed_time(e1) for e0, e1 in evs) / ksteps
        stack = {"kernel": "stack_decode_kernel", "us_per_launch": k_ms * 1e3, "bytes_per_launch": bytes_per_step,
                 "gbs": bytes_per_step / (k_ms * 1e-3) / 1e9, "launches_timed": ksteps, "layers_per_launch": L}
        ms = ms_stack
    ms, ms_e2e, ms_layers = max_over_ranks([ms, ms_e2e, ms_layers])

    # each expert kernel timed on its own (events around its launch, every layer)
    calls = [(handles[l], x, T, ys[l]) for l in range(L)]
    ksteps = max(3, min(args.steps, 10))
    kern = {}
    kernels = ((("gateup_nvfp4_kernel", K_GATE_UP, NV_GATE_UP_BYTES), ("down_nvfp4_kernel", K_DOWN, NV_DOWN_BYTES))
               if nv else (("gateup_mma_kernel", K_GATE_UP, GATE_UP_BYTES), ("down_mma_kernel", K_DOWN, DOWN_BYTES)))
    for kname, kid, per_exp in kernels:
        d = kernel_durations(flint, torch, stream, calls, kid, ksteps)
        tot_ms = sum(sum(r) for r in d)
        tot_bytes = ksteps * sum((u + 1) * per_exp for u in uniq)
        kern[kname] = {"us_per_launch": tot_ms * 1e3 / (ksteps * L), "bytes_per_launch": tot_bytes / (ksteps * L),
                       "gbs": tot_bytes / (tot_ms * 1e-3) / 1e9, "launches_timed": ksteps * L}
    dom = max(kern, key=lambda k: kern[k]["us_per_launch"])

    us_layer = ms * 1e3 / L
    achieved = bytes_per_step / (ms * 1e-3) / 1e9
    peak_hbm = float(pk["hbm_gbs"])
    if stack is not None:
        roof = {"bound": "hbm", **hbm_roof(stack["gbs"], peak_hbm, pk_kind),
                "traffic": traffic_from_profiles("stack_decode_kernel", name),
                "kernel": "stack_decode_kernel", "bytes_per_launch": stack["bytes_per_launch"],
                "us_per_launch": stack["us_per_launch"],
                "what": f"algorithmic bytes per launch (all {L} layers: unique touched experts incl. the shared one, "
                        f"{per_expert:,} B each) / its device duration (CUDA events around the launch, "
                        f"{stack['launches_timed']} extra launches)"}
    else:
        roof = {"bound": "hbm", **hbm_roof(kern[dom]["gbs"], peak_hbm, pk_kind),
                "traffic": traffic_from_profiles(dom, name),
                "kernel": dom, "bytes_per_launch": kern[dom]["bytes_per_launch"],
                "us_per_launch": kern[dom]["us_per_launch"],
                "what": "algorithmic bytes per launch (unique touched experts incl. the shared one x the matrices "
                        "this kernel reads) / its device duration (CUDA events around its launch in every layer of "
                        f"{ksteps} extra direct steps)"}
    line = {
        "metric": f"MoE-layer tokens/s, {'NVFP4 ' if nv else ''}decode stack T={T}",
        "value": whole_job_rate(L * T, ws, ms), "unit": "layer-tokens/s", "ms_per_step": ms,
        "us_per_layer": us_layer, "us_per_layer_no_graph": ms_direct * 1e3 / L,
        "dtype": "nvfp4 weights (e2m1 + e4m3 block scales), bf16 activations, f32 accumulation" if nv else "bf16",
        "config": {"workload": f"decode stack: {L} distinct {'NVFP4 (W4A16)' if nv else 'BF16'} MoE layers (H=2048, "
                               f"I=512, 256 routed + 1 shared, top-6 sigmoid, router bias N(0,0.5)), T={T} tokens "
                               f"({wl['x']} x, seed {wl['x_seed']})",
                   "weights_resident_gb": round(L * 257 * per_expert / 1e9, 2),
                   "l2": "inputs larger than L2 (each layer's weights are read once per step)",
                   "parallelism": f"replicas x{ws}", "graph": True},
        "unique_experts_per_layer": {"mean": float(np.mean(uniq)), "min": int(min(uniq)), "max": int(max(uniq))},
        "roofline": roof,
        "kernels": kern,
        "layer_hbm": {**hbm_roof(achieved, peak_hbm, pk_kind),
                      "what": "unique touched expert-weight bytes per layer / us per layer in the timed graph " +
                              ("(one persistent launch for the whole stack)" if stack is not None else
                               "(router, gate/up and down kernels chained by programmatic launch)")},
        "path": ("flint_moe_forward_layers: one persistent launch per step" if stack is not None else
                 f"{L} flint_moe_forward calls per step (3 kernels each, programmatic launch)"),
        "gpu_launches": (1 if stack is not None else 3 * L) * args.steps,
        "clocks": clocks,
        "e2e": {"value": whole_job_rate(L * T, ws, ms_e2e), "unit": "layer-tokens/s",
                "h2d_bytes_per_step": T * 2048 * 2, "d2h_bytes_per_step": L * T * 2048 * 2},
    }
    if stack is not None:
        line["stack_kernel"] = stack
        line["per_layer_calls"] = {
            "us_per_layer": ms_layers * 1e3 / L, "value": whole_job_rate(L * T, ws, ms_layers),
            "layer_hbm": hbm_roof(bytes_per_step / (ms_layers * 1e-3) / 1e9, peak_hbm, pk_kind),
            "kernels": kern,
            "what": f"the same stack as {L} flint_moe_forward calls per step (router, gate/up, down kernels), "
                    "replayed as one graph"}
    if rank == 0 and ws == 1 and cpu_seconds > 0:
        line["cpu_baseline"] = cpu_baseline(wl, layers[:2], cpu_seconds)
    return line


def bench_prefill(args, wl, lw, h, ws, rank, cpu_seconds, q=None):
    """One MoE layer (layer 0 of the stack: skewed router bias) on T = 8192
    tokens; weights (1.6 GB bf16, 0.45 GB NVFP4) exceed L2, so each step
    streams them again.  q: the NVFP4 encoding of the layer (NVFP4 handle)."""
    nv = q is not None
    import numpy as np
    import torch
    from sparse_moe_transformer_03_b300 import flint

    T = wl["T"]
    pk, pk_kind = peaks()
    xb = x_bits_for(wl)
    x = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).cuda()
    y = torch.empty_like(x)
    stream = torch.cuda.Stream()

    def step():
        flint.flint_moe_forward(h, x, T, y, stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    stream.synchronize()
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(torch.cuda.current_device()) as clk:
        with torch.cuda.stream(stream):
            ms = timed_ms(torch, stream, step, args.steps)
    torch.cuda.synchronize()
    clocks = clk.summary()

    x_host = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).pin_memory()
    y_host = torch.empty_like(x_host).pin_memory()
    x_dev = torch.empty_like(x)

    def step_e2e():
        x_dev.copy_(x_host, non_blocking=True)
        flint.flint_moe_forward(h, x_dev, T, y, stream)
        y_host.copy_(y, non_blocking=True)

    with torch.cuda.stream(stream):
        step_e2e()
        ms_e2e = timed_ms(torch, stream, step_e2e, max(3, args.steps // 2))
    ms, ms_e2e = max_over_ranks([ms, ms_e2e])
    # the dominant kernels timed on their own (events around each launch)
    ksteps = max(3, min(args.steps, 10))
    calls = [(h, x, T, y)]
    slots = 7 * T
    gu_flops, dn_flops = 2.0 * slots * 2048 * 1024, 2.0 * slots * 512 * 2048
    # algorithmic bytes: every expert's matrices once (all 257 are touched at this T), the activations
    # the kernel reads once and the outputs it writes once
    gu_w, dn_w = (NV_GATE_UP_BYTES, NV_DOWN_BYTES) if nv else (GATE_UP_BYTES, DOWN_BYTES)
    gu_bytes = 257 * gu_w + T * 2048 * 2 + slots * 512 * 2
    dn_bytes = 257 * dn_w + slots * 512 * 2 + slots * 2048 * 2
    sfx = "_nvfp4" if nv else ""
    kern = {}
    for kname, kid, fl, by in ((f"prefill_gateup{sfx}_kernel", K_GATE_UP, gu_flops, gu_bytes),
                               (f"prefill_down{sfx}_kernel", K_DOWN, dn_flops, dn_bytes)):
        d = kernel_durations(flint, torch, stream, calls, kid, ksteps)
        us = sum(r[0] for r in d) * 1e3 / ksteps
        kern[kname] = {"us_per_launch": us, "flops_per_launch": fl, "bytes_per_launch": by,
                       "tflops": fl / (us * 1e-6) / 1e12, "gbs": by / (us * 1e-6) / 1e9, "launches_timed": ksteps}
    dom = max(kern, key=lambda k: kern[k]["us_per_launch"])
    peak_hbm = float(pk["hbm_gbs"])
    peak_tc = float(pk["bf16_tflops"])
    kd = kern[dom]
    # the binding resource of the kernel's own roofline: the larger of bytes / bandwidth and flops / peak
    hbm_bound = kd["bytes_per_launch"] / peak_hbm / 1e9 >= kd["flops_per_launch"] / peak_tc / 1e12
    if hbm_bound:
        roof = {"bound": "hbm", **hbm_roof(kd["gbs"], peak_hbm, pk_kind)}
    else:
        roof = {"bound": "tensor", "achieved": kd["tflops"], "peak": peak_tc, "unit": "TFLOP/s",
                "frac": kd["tflops"] / peak_tc}
    roof.update({"traffic": traffic_from_profiles(dom, "nvfp4_prefill8192" if nv else "prefill8192"), "kernel": dom,
                 "us_per_launch": kd["us_per_launch"], "bytes_per_launch": kd["bytes_per_launch"],
                 "flops_per_launch": kd["flops_per_launch"], "tensor_frac": kd["tflops"] / peak_tc,
                 "what": f"algorithmic bytes and flops per launch / its device duration (CUDA events around its "
                         f"launch, {ksteps} extra direct steps); peaks = {pk_kind} HBM copy bandwidth and bf16 "
                         "burst; bound = the larger of bytes/bandwidth and flops/peak"})
    flops = FLOPS_PER_TOKEN * T
    achieved = flops / (ms * 1e-3) / 1e12
    line = {
        "metric": f"MoE-layer tokens/s, prefill T={T}", "value": whole_job_rate(T, ws, ms), "unit": "tokens/s",
        "ms_per_step": ms, "us_per_layer": ms * 1e3,
        "dtype": ("nvfp4 weights (e2m1 + e4m3 block scales) dequantised to bf16 in shared memory, bf16 activations, "
                  "f32 accumulation") if nv else "bf16",
        "config": {"workload": f"prefill: one {'NVFP4 (W4A16)' if nv else 'BF16'} MoE layer (H=2048, I=512, 256 routed "
                               f"+ 1 shared, top-6 sigmoid, router bias N(0,0.5)), T={T} tokens (x ~ N(0,1) "
                               f"RMS-normalised, seed {wl['x_seed']})",
                   "l2": f"inputs larger than L2 ({'0.45' if nv else '1.6'} GB of expert weights per step)",
                   "parallelism": f"replicas x{ws}"},
        "roofline": roof,
        "kernels": kern,
        "layer_tensor": {"achieved": achieved, "peak": peak_tc, "unit": "TFLOP/s", "frac": achieved / peak_tc,
                         "peak_kind": f"{pk_kind} dense bf16 (burst)",
                         "what": f"dense layer FLOPs (experts {7 * 6 * 2048 * 512 * T / 1e9:.1f} GFLOP + router "
                                 f"{2 * 256 * 2048 * T / 1e9:.1f}) / step time"},
        "gpu_launches": 6 * args.steps,
        "clocks": clocks,
        "e2e": {"value": whole_job_rate(T, ws, ms_e2e), "unit": "tokens/s", "h2d_bytes_per_step": T * 2048 * 2,
                "d2h_bytes_per_step": T * 2048 * 2},
    }
    if rank == 0 and ws == 1 and cpu_seconds > 0:
        line["cpu_baseline"] = cpu_baseline_prefill(wl, lw, xb, cpu_seconds, q)
    return line


def build_lm_head(flint, device, V, seed):
    """A seeded bf16 head [V][2048] quantised to NVFP4 on the device and its
    handle; returns (handle, host packed, host scales, tensor scale)."""
    import torch
    from synth import gen
    w = torch.empty((V, gen.H), dtype=torch.bfloat16, device="cuda")
    device.fill_normal_bf16(w, seed, 0, gen.T_LM_HEAD, gen.WEIGHT_STD)
    pk, sc, ts = device.nvfp4_quantize(w)
    del w
    t = float(ts[0].item())
    h = flint.flint_lm_head_create((pk[0], sc[0], t), V)
    parts = (pk[0][:LM_HEAD_SAMPLE_ROWS].cpu().numpy(), sc[0][:LM_HEAD_SAMPLE_ROWS].cpu().numpy(), t)
    del pk, sc
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return h, parts


def bench_lm_head(args, wl, ws, rank, cpu_seconds):
    """The 4-bit output layer: one flint_lm_head_forward per step on a
    V x 2048 NVFP4 head (151 MB, larger than L2, so each step streams it)."""
    import numpy as np
    import torch
    from sparse_moe_transformer_03_b300 import flint
    from synth import device

    T, V = wl["T"], LM_HEAD_V
    pk_, pk_kind = peaks()
    h, parts = build_lm_head(flint, device, V, LM_HEAD_SEED)
    xb = x_bits_for(wl)
    x = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).cuda()
    logits = torch.empty((T, V), dtype=torch.float32, device="cuda")
    stream = torch.cuda.Stream()

    def step():
        flint.flint_lm_head_forward(h, x, T, logits, stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    stream.synchronize()
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(torch.cuda.current_device()) as clk:
        with torch.cuda.stream(stream):
            ms = timed_ms(torch, stream, step, args.steps)
    torch.cuda.synchronize()
    clocks = clk.summary()
    x_host = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).pin_memory()
    l_host = torch.empty((T, V), dtype=torch.float32).pin_memory()
    x_dev = torch.empty_like(x)

    def step_e2e():
        x_dev.copy_(x_host, non_blocking=True)
        flint.flint_lm_head_forward(h, x_dev, T, logits, stream)
        l_host.copy_(logits, non_blocking=True)

    with torch.cuda.stream(stream):
        step_e2e()
        ms_e2e = timed_ms(torch, stream, step_e2e, max(3, args.steps // 2))
    ms, ms_e2e = max_over_ranks([ms, ms_e2e])
    flint.flint_lm_head_destroy(h)
    # algorithmic bytes: every code and block scale once, x once, the logits written once
    w_bytes = V * (2048 // 2 + 2048 // 16)
    by = w_bytes + T * 2048 * 2 + T * V * 4
    gbs = by / (ms * 1e-3) / 1e9
    line = {
        "metric": f"output-layer tokens/s, NVFP4 lm_head T={T}", "value": whole_job_rate(T, ws, ms),
        "unit": "tokens/s", "ms_per_step": ms, "us_per_call": ms * 1e3,
        "dtype": "nvfp4 weights (e2m1 + e4m3 block scales), bf16 activations, f32 accumulation and logits",
        "config": {"workload": f"output layer: NVFP4 (W4A16) head [{V}][2048] (vocabulary assumed; the pages give "
                               f"none), T={T} tokens ({wl['x']} x, seed {wl['x_seed']})",
                   "l2": "inputs larger than L2 (151 MB of head weights per step)", "parallelism": f"replicas x{ws}"},
        "roofline": {"bound": "hbm", **hbm_roof(gbs, float(pk_["hbm_gbs"]), pk_kind),
                     "traffic": traffic_from_profiles("lm_head_nvfp4_kernel", wl["name"]),
                     "kernel": "lm_head_nvfp4_kernel", "bytes_per_launch": by, "us_per_launch": ms * 1e3,
                     "what": "algorithmic bytes per launch (V x 1152 bytes of codes and scales + x + the fp32 logits "
                             "written) / its device duration (CUDA events around each step's single launch)"},
        "gpu_launches": args.steps,
        "clocks": clocks,
        "e2e": {"value": whole_job_rate(T, ws, ms_e2e), "unit": "tokens/s", "h2d_bytes_per_step": T * 2048 * 2,
                "d2h_bytes_per_step": T * V * 4},
    }
    if rank == 0 and ws == 1 and cpu_seconds > 0:
        line["cpu_baseline"] = cpu_baseline_lm_head(wl, xb, parts, cpu_seconds)
    return line


def cpu_baseline_lm_head(wl, xb, parts, seconds):
    """The oracle, as it stands, on the head's first LM_HEAD_SAMPLE_ROWS rows,
    scaled to the full vocabulary."""
    import oracle
    pk, sc, ts = parts
    m = oracle.Mat(packed=pk, scales=sc, tensor_scale=ts)
    t0 = time.perf_counter()
    reps = 0
    while True:
        oracle.lm_head(xb, m)
        reps += 1
        if time.perf_counter() - t0 > seconds or reps >= 20:
            break
    dt = (time.perf_counter() - t0) / reps * LM_HEAD_V / LM_HEAD_SAMPLE_ROWS
    return {"value": wl["T"] / dt, "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"first {LM_HEAD_SAMPLE_ROWS} of the {LM_HEAD_V} rows at T={wl['T']}, {reps} reps, "
                      f"scaled by {LM_HEAD_V // LM_HEAD_SAMPLE_ROWS} to the whole head"}


COMMON_KEYS = ("n_gpus", "steps", "warmup", "higher_is_better", "scaling", "vs_baseline", "data")


def run_flint(args, ws, rank, local):
    """The flint arm.  --workload all (the default): the BF16 decode stack at
    T = 1 (the headline line), then T = 8 and 32, the T = 8192 prefill on the
    stack's first layer, the NVFP4 stack at T = 1, 8 and 32 and the NVFP4
    T = 8192 prefill, each as an entry of the line's "configs"; otherwise the
    named workload alone."""
    import torch
    from sparse_moe_transformer_03_b300 import flint
    from synth import device

    flint.load_library()
    device.build()
    names = ALL_ORDER if args.workload == "all" else [args.workload]
    L = args.layers
    results = {}
    t_gen = time.perf_counter()
    bf16_names = [n for n in names if not WORKLOADS[n].get("nvfp4") and not WORKLOADS[n].get("lm_head")]
    nv_names = [n for n in names if WORKLOADS[n].get("nvfp4")]
    lh_names = [n for n in names if WORKLOADS[n].get("lm_head")]
    gen_s = {}
    if bf16_names:
        layers, handles = build_bf16_stack(flint, device, L if any(not WORKLOADS[n].get("prefill") for n in bf16_names)
                                           else 1)
        gen_s["bf16"] = round(time.perf_counter() - t_gen, 2)
        for n in bf16_names:
            wl = WORKLOADS[n]
            cpu_s = HEADLINE_CPU_SECONDS if n == names[0] else CONFIG_CPU_SECONDS
            if wl.get("prefill"):
                results[n] = bench_prefill(args, wl, layers[0], handles[0], ws, rank, cpu_s)
            else:
                results[n] = bench_decode(args, wl, n, layers, handles, ws, rank, False, cpu_s)
        for h in handles:
            flint.flint_moe_destroy(h)
        del layers, handles
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    if nv_names:
        t0 = time.perf_counter()
        layers, handles = build_nvfp4_stack(flint, device, L if any(not WORKLOADS[n].get("prefill") for n in nv_names)
                                            else 1)
        gen_s["nvfp4"] = round(time.perf_counter() - t0, 2)
        for n in nv_names:
            wl = WORKLOADS[n]
            cpu_s = HEADLINE_CPU_SECONDS if n == names[0] else CONFIG_CPU_SECONDS
            if wl.get("prefill"):
                results[n] = bench_prefill(args, wl, layers[0][0], handles[0], ws, rank, cpu_s, layers[0][1])
            else:
                results[n] = bench_decode(args, wl, n, layers, handles, ws, rank, True, cpu_s)
        for h in handles:
            flint.flint_moe_destroy(h)
        del layers, handles
        torch.cuda.empty_cache()

    for n in lh_names:
        cpu_s = HEADLINE_CPU_SECONDS if n == names[0] else CONFIG_CPU_SECONDS
        results[n] = bench_lm_head(args, dict(WORKLOADS[n], name=n), ws, rank, cpu_s)
        torch.cuda.empty_cache()

    head = dict(results[names[0]])
    line = {"metric": head.pop("metric"), "value": head.pop("value"), "unit": head.pop("unit"),
            "n_gpus": ws, "steps": args.steps, "warmup": args.warmup, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            "data": "synthetic (seeded counter-based generator; random-init weights)"}
    line.update(head)
    line["gen_seconds"] = gen_s
    if len(names) > 1:
        line["configs"] = {n: results[n] for n in names[1:]}
        line["gpu_launches"] = sum(r["gpu_launches"] for r in results.values())
        line["gpu_launches_headline"] = results[names[0]]["gpu_launches"]
    if rank == 0:
        print(json.dumps(line), flush=True)


ALL_ORDER = ["decode1", "decode8", "decode32", "prefill8192", "nvfp4_decode1", "nvfp4_decode8", "nvfp4_decode32",
             "nvfp4_prefill8192", "nvfp4_lm_head1", "nvfp4_lm_head32"]
HEADLINE_CPU_SECONDS = 10.0
CONFIG_CPU_SECONDS = 4.0


def main():
    args = parse()
    ws, rank, local = dist_setup(args)
    if args.impl == "reference":
        wl = dict(WORKLOADS["decode1" if args.workload == "all" else args.workload])
        run_reference(args, wl, ws, rank)
    else:
        run_flint(args, ws, rank, local)
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
