"""Throughput of the fused NVFP4 activation producers on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step is one call of the fused RMSNorm + AdaLN -> NVFP4 producer over the
65,280 x 7,168 bf16 workload (32 frames x 2,040 tokens, the MiniMax-H3 video
DiT shape).  The headline is HBM GB/s: the algorithmic bytes of a call (bf16
input read once, codes and swizzled scales written once, gamma and the
modulation table read once) over the call's device time.  The input (936 MB)
is larger than L2, so nothing is flushed between steps.

Printed as one JSON line on rank 0, with:
  roofline     the producer kernel against the measured HBM copy bandwidth,
               and its DRAM traffic per launch from the committed ncu summary
  cpu_baseline the CPU oracle on the host cores over a bounded sample
  e2e          the same metric through the public call with host buffers:
               pinned host -> device copy of the step's inputs, the call, and
               device -> host copy of its codes and scales, all timed
  producers    the other producers measured the same way (SwiGLU, the
               standalone quantize, the attention-output quantize)
  clocks       nvidia-smi samples taken while the kernels ran

Under torchrun (N > 1) every rank runs its own copy of the workload (the rows
are independent and the global scale is static, so no data moves between
ranks); the time is the maximum over ranks and the value counts all ranks'
bytes.  ``--impl reference`` times the CPU oracle instead (rank 0 only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import re
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import workloads  # noqa: E402

METRIC = "fused RMSNorm+AdaLN→NVFP4 HBM GB/s (% of GB300 peak) at 65,280×7,168 bf16"
ROWS, COLS = workloads.TOKENS, workloads.HIDDEN
FRAMES, RPF = workloads.FRAMES, workloads.TOKENS_PER_FRAME
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 2**20


# --------------------------------------------------------------------------- #
# bytes and peaks                                                               #
# --------------------------------------------------------------------------- #

def padded(rows: int) -> int:
    return (rows + 127) // 128 * 128


def out_bytes(rows: int, cols: int) -> int:
    return rows * cols // 2 + padded(rows) * cols // 16


def adaln_bytes(rows: int, cols: int, frames: int) -> int:
    # x read + codes + scales written + gamma + modulation table + global scale
    return 2 * rows * cols + out_bytes(rows, cols) + 2 * cols + frames * 2 * cols * 2 + 4


def quantize_bytes(rows: int, cols: int) -> int:
    return 2 * rows * cols + out_bytes(rows, cols) + 4


def swiglu_bytes(rows: int, cols: int) -> int:
    return 4 * rows * cols + out_bytes(rows, cols) + 4


def residual_bytes(rows: int, cols: int, frames: int) -> int:
    # h read and written (fp32), o read, codes + scales, bias + gamma, gate and modulation tables
    return (4 + 4 + 2) * rows * cols + out_bytes(rows, cols) + 2 * 2 * cols + frames * 3 * cols * 2 + 4


def qkv_bytes(rows: int, heads: int, head_dim: int, rot: int) -> int:
    # q, k, v read and written (bf16), their biases, the cos and sin tables
    d = heads * head_dim
    return 3 * 2 * rows * d * 2 + 3 * d * 2 + 2 * rows * rot * 2


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


# NVFP4 dense tensor rate over bf16 dense (nominal 13.5 / 2.25 PFLOP/s per GB300).
FP4_OVER_BF16 = 6.0
FALLBACK_BF16_TFLOPS = 1900.0


def fp4_peak():
    """The NVFP4 dense tensor peak in TFLOP/s: the measured cuBLAS bf16 burst rate
    times the nominal FP4:bf16 ratio (no FP4 rate is measured on the pool)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]) * FP4_OVER_BF16, "measured bf16 burst x 6 (13.5/2.25 nominal)"
    except (OSError, KeyError, ValueError):
        return FALLBACK_BF16_TFLOPS * FP4_OVER_BF16, "fallback bf16 x 6"


# The sources each kernel is compiled from (its own file and the shared device header).
KERNEL_SOURCES = {
    "adaln_block_kernel": ("adaln.cu", "h3q_device.cuh"),
    "swiglu_kernel": ("swiglu.cu", "h3q_device.cuh", "h3q_silu.cuh"),
    "swiglu_ring_kernel": ("swiglu.cu", "h3q_device.cuh", "h3q_silu.cuh"),
    "gemm_swiglu_kernel": ("gemm_swiglu.cu", "h3q_device.cuh", "h3q_silu.cuh", "h3q_async.cuh"),
    "quantize_kernel": ("quantize.cu", "h3q_device.cuh"),
}


def _code_only(text: str) -> str:
    """C/CUDA source without its comments and whitespace (string literals in
    these sources hold no comment markers), so comment edits keep a record."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return "".join(text.split())


def kernel_source_hash(kernel: str) -> str:
    """Hash of the code (comments and whitespace stripped) of the sources a
    kernel is compiled from: records taken from a kernel stay valid until its
    code changes."""
    csrc = os.path.join(ROOT, "nvfp4_activation_quantize_gb300", "csrc")
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(csrc, name)) as f:
            h.update(name.encode() + b"\0" + _code_only(f.read()).encode())
    return h.hexdigest()[:16]


def recorded_value(kernel: str, path: str):
    """The number recorded for `kernel` in a profiles/ record (lines: kernel
    source-hash value), if it was taken from the current kernel sources."""
    if not os.path.exists(path):
        return None
    want = kernel_source_hash(kernel)
    with open(path) as f:
        for line in f:
            parts = line.split()
            if len(parts) >= 3 and not line.startswith("#") and parts[0] == kernel:
                return float(parts[2]) if parts[1] == want else None
    return None


def recorded_traffic(kernel: str, path: str | None = None):
    """DRAM bytes per launch of `kernel` from profiles/dram_traffic.txt, if they were
    taken from the current kernel sources (lines: kernel source-hash bytes)."""
    v = recorded_value(kernel, path or os.path.join(ROOT, "profiles", "dram_traffic.txt"))
    return None if v is None else int(v)


# --------------------------------------------------------------------------- #
# clocks                                                                        #
# --------------------------------------------------------------------------- #

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while kernels run."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self._reader = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self._reader = threading.Thread(target=self._read, daemon=True)
        self._reader.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.monotonic(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self._reader.join(timeout=5)

    def summary(self, t0: float, t1: float):
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for t, line in self.lines:
            if not (t0 <= t <= t1):
                continue
            f = [p.strip() for p in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower() in ("active", "0x1", "1"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm.sort()
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# --------------------------------------------------------------------------- #
# timing helpers                                                                #
# --------------------------------------------------------------------------- #

def memcpy_d2d_ceiling(dev, stream, nbytes: int = 4 << 30, reps: int = 10) -> dict:
    """A plain device-to-device copy (torch's copy_ of a contiguous buffer, a
    cudaMemcpyAsync) of `nbytes`, read and written once per copy: the bandwidth a
    copy reaches on this GPU, next to the producers' algorithmic GB/s."""
    src = torch.empty(nbytes, dtype=torch.uint8, device=dev).fill_(1)
    dst = torch.empty_like(src)
    with torch.cuda.stream(stream):
        for _ in range(3):
            dst.copy_(src)
    _, per = time_launches(lambda: dst.copy_(src), reps, stream)
    ms = sorted(per)[len(per) // 2]
    del src, dst
    torch.cuda.empty_cache()
    return {"gbs": round(2 * nbytes / (ms * 1e-3) / 1e9, 1), "bytes_copied": nbytes, "median_ms": round(ms, 4),
            "copies": reps}


def time_launches(fn, steps: int, stream, flush=None):
    """Run fn() `steps` times on `stream`, each bracketed by its own CUDA events.
    Returns (total_ms from the first start to the last end, per-launch ms list)."""
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    with torch.cuda.stream(stream):
        for i in range(steps):
            if flush is not None:
                flush()
            starts[i].record(stream)
            fn()
            ends[i].record(stream)
    torch.cuda.synchronize()
    per = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    return starts[0].elapsed_time(ends[-1]), per


def max_over_ranks(ms: float, world: int, device) -> float:
    """The slowest rank's elapsed milliseconds: a replica run's timed region ends
    when its last rank ends (all-reduce MAX; the identity on one rank)."""
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    if world > 1:
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_gbs(bytes_per_rank_step: float, steps: int, world: int, ms: float) -> float:
    """Whole-job GB/s: the bytes every rank processed over `steps` steps in `ms`."""
    return world * bytes_per_rank_step * steps / (ms * 1e-3) / 1e9


def calibrate_adaln_gsf(w) -> float:
    """Global scale from max |modulated x| (torch fp32 on the GPU, a calibration
    pass outside the timed region)."""
    x, gamma, table = w["x"], w["gamma"].float(), w["table"].float()
    amax = 0.0
    step = 4096
    for r0 in range(0, x.shape[0], step):
        xf = x[r0:r0 + step].float()
        rstd = torch.rsqrt(xf.pow(2).mean(1, keepdim=True) + w["eps"])
        t = torch.arange(r0, r0 + xf.shape[0], device=x.device) // w["rows_per_frame"]
        y = xf * rstd * gamma * (1 + table[t, 1]) + table[t, 0]
        amax = max(amax, float(y.abs().max()))
    return 2688.0 / amax


def calibrate_swiglu_gsf(gate, up) -> float:
    amax = 0.0
    for r0 in range(0, gate.shape[0], 4096):
        g = gate[r0:r0 + 4096].float()
        y = torch.nn.functional.silu(g) * up[r0:r0 + 4096].float()
        amax = max(amax, float(y.abs().max()))
    return 2688.0 / amax


def gemm_operands(h3q, dev, stream, rows: int, hidden: int = COLS, ffn: int = workloads.FFN, seed: int = 8):
    """The FFN-up GEMM's NVFP4 operands (the activation and the value/gate-paired
    weight quantized by the library's own quantize), alpha, and the output's global
    scale from a calibration launch's y (torch abs-max), all outside any timed
    region.  Returns (operands tuple for h3q_gemm_swiglu_nvfp4, flops per launch)."""
    w = workloads.ffn_up_inputs(dev, rows=rows, hidden=hidden, ffn=ffn, seed=seed)
    ops = []
    gs = []
    for t in (w["x"], w["w"]):
        g = 2688.0 / float(t.abs().max().float())
        c, sc = h3q.h3q_quantize_nvfp4(t, torch.tensor([g], dtype=torch.float32, device=dev), stream=stream)
        ops += [c, sc]
        gs.append(g)
    del w
    alpha = torch.tensor([1.0 / (gs[0] * gs[1])], dtype=torch.float32, device=dev)
    y = torch.empty((rows, ffn), dtype=torch.bfloat16, device=dev)
    one = torch.ones(1, dtype=torch.float32, device=dev)
    h3q.h3q_gemm_swiglu_nvfp4(ops[0], ops[1], ops[2], ops[3], alpha, one, y=y, stream=stream)
    gsf = torch.tensor([2688.0 / float(y.abs().max().float())], dtype=torch.float32, device=dev)
    del y
    return (ops[0], ops[1], ops[2], ops[3], alpha, gsf), 2 * rows * 2 * ffn * hidden


# --------------------------------------------------------------------------- #
# our arm                                                                       #
# --------------------------------------------------------------------------- #

def workload_config() -> dict:
    """The headline workload, named the same way by both arms."""
    return {"workload": f"rmsnorm_adaln_nvfp4 {ROWS}x{COLS} bf16, {FRAMES} frames x {RPF} tokens, "
                        "per-channel LogNormal(0,0.5) scales",
            "rows": ROWS, "cols": COLS, "frames": FRAMES, "rows_per_frame": RPF}


def run_ours(args, rank, world, dev):
    import nvfp4_activation_quantize_gb300 as h3q

    h3q.library()
    stream = torch.cuda.current_stream(dev)
    w = workloads.adaln_inputs(dev)
    gsf_val = calibrate_adaln_gsf(w)
    gsf = torch.tensor([gsf_val], dtype=torch.float32, device=dev)
    codes = torch.empty((ROWS, COLS // 2), dtype=torch.uint8, device=dev)
    scales = torch.empty((padded(ROWS), COLS // 16), dtype=torch.uint8, device=dev)

    def step():
        h3q.h3q_rmsnorm_adaln_nvfp4(w["x"], w["gamma"], w["table"], gsf, rows_per_frame=RPF,
                                    eps=w["eps"], codes=codes, scales=scales, stream=stream)

    sampler = ClockSampler(dev.index if dev.index is not None else 0)
    sampler.start()
    for _ in range(args.warmup):
        step()
    # keep the GPU busy long enough for the clock samples (untimed)
    torch.cuda.synchronize()
    soak_t0 = time.monotonic()
    while time.monotonic() - soak_t0 < args.soak:
        for _ in range(50):
            step()
        torch.cuda.synchronize()

    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t0 = time.monotonic()
    total_ms, per = time_launches(step, args.steps, stream)
    t1 = time.monotonic()
    if world > 1:
        torch.distributed.barrier()
    sampler.stop()
    clocks = sampler.summary(soak_t0, t1)

    total_ms = max_over_ranks(total_ms, world, dev)
    nbytes = adaln_bytes(ROWS, COLS, FRAMES)
    value = job_gbs(nbytes, args.steps, world, total_ms)
    launch_ms = sum(per) / len(per)
    achieved = nbytes / (launch_ms * 1e-3) / 1e9
    peak, peak_kind = hbm_peak()

    result = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(total_ms / args.steps, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": {
            **workload_config(),
            "l2": f"inputs larger than L2 ({2 * ROWS * COLS / 1e6:.0f} MB bf16 read per step); no flush",
            "algorithmic_bytes_per_step": nbytes,
            "rows_per_s": round(world * ROWS * args.steps / (total_ms * 1e-3)),
            "global_scale": gsf_val,
            "soak_s": args.soak,
            "parallelism": f"replica x{world}" if world > 1 else "single GPU",
        },
        "roofline": {
            "bound": "hbm",
            "achieved": round(achieved, 1),
            "peak": peak,
            "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "traffic": recorded_traffic("adaln_block_kernel"),
            "peak_source": f"{peak_kind} HBM copy bandwidth (MEASURED_PEAKS.json hbm_gbs)"
                           if peak_kind == "measured" else "fallback 6.8 TB/s",
            "kernel": "adaln_block_kernel<448, 7> (7,168 columns, one 448-thread CTA per SM)",
            "launch_ms": round(launch_ms, 5),
        },
        "gpu_launches": args.steps,
        "clocks": clocks,
    }

    if rank == 0 and world == 1 and not args.no_extras:
        args.sm_mhz_seen = clocks.get("sm_mhz") or clocks.get("sm_max_mhz") or 2070.0
        result["roofline"]["memcpy_d2d"] = memcpy_d2d_ceiling(dev, stream)
        ipe = recorded_value("adaln_block_kernel", os.path.join(ROOT, "profiles", "inst_per_element.txt"))
        if ipe is not None:
            props = torch.cuda.get_device_properties(dev)
            ms_issue = ROWS * COLS * ipe / (props.multi_processor_count * 4 * 32 * args.sm_mhz_seen * 1e6) * 1e3
            result["roofline"]["issue_ceiling"] = {
                "thread_inst_per_elem": ipe, "ms_at_full_issue": round(ms_issue, 4),
                "issue_efficiency": round(ms_issue / launch_ms, 3), "sm_mhz": args.sm_mhz_seen,
                "source": "ncu smsp__sass_thread_inst_executed.sum per element, profiles/inst_per_element.txt"}
        result["producers"] = measure_producers(h3q, dev, stream, args)
        result["e2e"] = measure_e2e(h3q, dev, stream, w, gsf, args)
        if not args.no_cpu_baseline:
            result["cpu_baseline"] = cpu_baseline(seconds=args.cpu_seconds)
    elif world > 1:
        result["e2e"] = measure_e2e(h3q, dev, stream, w, gsf, args, world=world)
    return result


def _cpulist(text: str) -> list[int]:
    """'0-3,8,10-11' -> [0, 1, 2, 3, 8, 10, 11]."""
    cpus = []
    for part in text.strip().split(","):
        if not part:
            continue
        lo, _, hi = part.partition("-")
        cpus.extend(range(int(lo), int(hi or lo) + 1))
    return cpus


def gpu_locality(dev) -> dict:
    """The GPU's PCI address, its NUMA node and the CPUs local to it, from sysfs
    (read only; {} where the files are missing)."""
    props = torch.cuda.get_device_properties(dev)
    try:
        bus = f"{props.pci_domain_id:04x}:{props.pci_bus_id:02x}:{props.pci_device_id:02x}.0"
    except AttributeError:
        return {}
    base = f"/sys/bus/pci/devices/{bus}"
    out = {"pci": bus}
    try:
        with open(f"{base}/numa_node") as f:
            out["numa_node"] = int(f.read().strip())
        with open(f"{base}/local_cpulist") as f:
            out["local_cpus"] = _cpulist(f.read())
    except OSError:
        pass
    return out


def pages_by_node(t: torch.Tensor) -> dict:
    """How the pages of a host tensor's mapping are spread over NUMA nodes
    (/proc/self/numa_maps: the mapping that contains its first byte)."""
    addr = t.data_ptr()
    try:
        with open("/proc/self/maps") as f:
            start = None
            for line in f:
                lo, hi = (int(v, 16) for v in line.split()[0].split("-"))
                if lo <= addr < hi:
                    start = lo
                    break
        if start is None:
            return {}
        with open("/proc/self/numa_maps") as f:
            for line in f:
                fields = line.split()
                if int(fields[0], 16) == start:
                    return {k: int(v) for k, v in (x.split("=") for x in fields[2:])
                            if k.startswith("N") and k[1:].isdigit()}
    except (OSError, ValueError):
        pass
    return {}


def measure_e2e(h3q, dev, stream, w, gsf, args, world=1):
    """Runs measure_e2e_placed with this thread (the one that allocates the pinned
    buffers and enqueues the copies) on the CPUs local to the GPU, so the pinned
    pages land on the GPU's own node; the placement is recorded."""
    loc = gpu_locality(dev)
    before = os.sched_getaffinity(0) if hasattr(os, "sched_getaffinity") else None
    cpus = [c for c in loc.get("local_cpus", []) if before is None or c in before]
    if cpus:
        os.sched_setaffinity(0, cpus)
    try:
        out = measure_e2e_placed(h3q, dev, stream, w, gsf, args, world)
    finally:
        if cpus and before is not None:
            os.sched_setaffinity(0, before)
    out["placement"] = {"gpu": loc, "affinity": cpus or (sorted(before) if before else None),
                        "x_pages_by_node": out.pop("_x_pages", {})}
    return out


def measure_e2e_placed(h3q, dev, stream, w, gsf, args, world=1):
    """The same metric through the C-ABI host-buffer call (h3q_rmsnorm_adaln_nvfp4_host,
    through HostPipeline): each step copies gamma and the modulation table from pinned
    host memory to the device, then the call copies x in, runs the producer and copies
    codes and scales back to pinned host memory, pipelined over 2,048-row chunks (the
    producer on the caller's stream, a library stream per copy direction).  The timed
    region (CUDA events on the caller's stream) covers every copy of the step."""
    from nvfp4_activation_quantize_gb300.host import HostPipeline

    hx = torch.empty(w["x"].shape, dtype=w["x"].dtype).pin_memory()
    hx.copy_(w["x"])
    hg = w["gamma"].cpu().pin_memory()
    ht = w["table"].cpu().pin_memory()
    hc = torch.empty((ROWS, COLS // 2), dtype=torch.uint8).pin_memory()
    hs = torch.empty((padded(ROWS), COLS // 16), dtype=torch.uint8).pin_memory()
    pipe = HostPipeline(dev, COLS, chunk_rows=2048)

    def step():
        pipe.rmsnorm_adaln_nvfp4(hx, hg, ht, gsf, hc, hs, rows_per_frame=RPF, eps=w["eps"])

    with torch.cuda.stream(stream):
        for _ in range(3):
            step()
    torch.cuda.synchronize()
    steps = max(3, min(args.steps, 10))
    total_ms, per_step = time_launches(step, steps, stream)
    total_ms = max_over_ranks(total_ms, world, dev)
    nbytes = adaln_bytes(ROWS, COLS, FRAMES)
    h2d = hx.numel() * 2 + hg.numel() * 2 + ht.numel() * 2
    d2h = hc.numel() + hs.numel()
    out = {
        "value": round(job_gbs(nbytes, steps, world, total_ms), 1),
        "unit": "GB/s",
        "h2d_bytes_per_step": h2d,
        "d2h_bytes_per_step": d2h,
        "steps": steps,
        "ms_per_step": round(total_ms / steps, 3),
        "call": "h3q_rmsnorm_adaln_nvfp4_host",
        "pipeline": {"chunk_rows": pipe.chunk_rows, "depth": pipe.depth, "streams": 3},
        "check": e2e_matches(h3q, dev, w, gsf, hc, hs),
        "_x_pages": pages_by_node(hx),
    }
    if world == 1:
        link = host_link(dev)
        bound = link_bound_ms(h2d, d2h, link)
        out["host_link"] = dict(link, bound_ms_per_step=round(bound, 3),
                                frac_of_link_bound=round(bound / (total_ms / steps), 3),
                                step_buffers=buffer_rates(dev, hx, hc))
        out["step_ms"] = [round(v, 3) for v in per_step]
        out["chunk_copies"] = chunk_copies(dev, hx, hc, hs, pipe.chunk_rows)
    return out


def chunk_copies(dev, hx, hc, hs, chunk_rows: int) -> dict:
    """The step's own copies without the producer: x host to device chunk by chunk
    on one stream, codes and scales device to host chunk by chunk on another, each
    direction alone and both at once (ms for the whole step's bytes).  Set beside
    the pipelined step's time, it tells a slow step whose copies are slow from one
    whose copies are fine but badly overlapped."""
    rows, quads = hx.shape[0], hx.shape[1] // 64
    dx = torch.empty((chunk_rows, hx.shape[1]), dtype=hx.dtype, device=dev)
    dc = torch.empty((chunk_rows, hc.shape[1]), dtype=hc.dtype, device=dev)
    ds = torch.empty(chunk_rows * hs.shape[1], dtype=hs.dtype, device=dev)
    hs_flat = hs.view(-1)
    s1, s2 = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def h2d():
        with torch.cuda.stream(s1):
            for r0 in range(0, rows, chunk_rows):
                n = min(chunk_rows, rows - r0)
                dx[:n].copy_(hx[r0:r0 + n], non_blocking=True)

    def d2h():
        with torch.cuda.stream(s2):
            for r0 in range(0, rows, chunk_rows):
                n = min(chunk_rows, rows - r0)
                pad_n = -(-n // 128) * 128
                hc[r0:r0 + n].copy_(dc[:n], non_blocking=True)
                o = r0 // 128 * quads * 512
                hs_flat[o:o + pad_n * hs.shape[1]].copy_(ds[:pad_n * hs.shape[1]], non_blocking=True)

    def timed(*fns, reps=3):
        res = []
        for _ in range(reps):
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            for fn in fns:
                fn()
            torch.cuda.synchronize()
            res.append((time.perf_counter() - t0) * 1e3)
        return round(min(res), 3)

    out = {"h2d_ms": timed(h2d), "d2h_ms": timed(d2h), "both_ms": timed(h2d, d2h)}
    del dx, dc, ds
    return out


def buffer_rates(dev, hx, hc, reps: int = 3) -> dict:
    """Plain copy rates of the step's own pinned buffers (x in, codes out), beside
    host_link's fresh buffers: a host buffer that copies slower than fresh pinned
    memory on the same box points at its backing, not at the pipeline."""
    dx = torch.empty(hx.shape, dtype=hx.dtype, device=dev)
    dc = torch.empty(hc.shape, dtype=hc.dtype, device=dev)

    def rate(fn, nbytes):
        fn()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(reps):
            fn()
        torch.cuda.synchronize()
        return round(reps * nbytes / (time.perf_counter() - t0) / 1e9, 1)

    res = {"x_h2d_gbs": rate(lambda: dx.copy_(hx, non_blocking=True), hx.numel() * hx.element_size()),
           "codes_d2h_gbs": rate(lambda: hc.copy_(dc, non_blocking=True), hc.numel())}
    del dx, dc
    return res


def host_link(dev, nbytes: int = 512 << 20, reps: int = 8) -> dict:
    """Pinned host <-> device copy bandwidth on this machine: each direction alone and
    both at once on two streams (GB/s per direction)."""
    h_in = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    h_out = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    d_in = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    d_out = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    s1, s2 = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def timed(fn, trials: int = 3):
        for _ in range(2):
            fn()
        rates = []
        for _ in range(trials):
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            for _ in range(reps):
                fn()
            torch.cuda.synchronize()
            rates.append(round(reps * nbytes / (time.perf_counter() - t0) / 1e9, 1))
        return rates

    def both():
        with torch.cuda.stream(s1):
            d_in.copy_(h_in, non_blocking=True)
        with torch.cuda.stream(s2):
            h_out.copy_(d_out, non_blocking=True)

    # each rate is the best of three trials (the link's capability); the two-way
    # trials are kept, since concurrent copies in both directions now and then run
    # at about half their usual rate on this platform
    h2d = timed(lambda: d_in.copy_(h_in, non_blocking=True))
    d2h = timed(lambda: h_out.copy_(d_out, non_blocking=True))
    two = timed(both)
    res = {"h2d_gbs": max(h2d), "d2h_gbs": max(d2h), "both_gbs_each": max(two), "both_gbs_trials": two,
           "bytes_per_copy": nbytes}
    del h_in, h_out, d_in, d_out
    return res


def link_bound_ms(h2d_bytes: int, d2h_bytes: int, link: dict) -> float:
    """The shortest step the host link allows: the smaller direction's bytes moved
    while the larger one runs beside it (both at the two-way rate), the rest of the
    larger direction alone."""
    big, small = (h2d_bytes, d2h_bytes) if h2d_bytes >= d2h_bytes else (d2h_bytes, h2d_bytes)
    big_rate = link["h2d_gbs"] if h2d_bytes >= d2h_bytes else link["d2h_gbs"]
    return (small / (link["both_gbs_each"] * 1e9) + (big - small) / (big_rate * 1e9)) * 1e3


def e2e_matches(h3q, dev, w, gsf, hc, hs) -> bool:
    """The host-buffer outputs equal the device-buffer call's, byte for byte."""
    c, s = h3q.h3q_rmsnorm_adaln_nvfp4(w["x"], w["gamma"], w["table"], gsf, rows_per_frame=RPF,
                                       eps=w["eps"])
    torch.cuda.synchronize()
    return bool(torch.equal(c.cpu(), hc) and torch.equal(s.cpu(), hs))


def measure_producers(h3q, dev, stream, args):
    """The other producers, each timed per launch with CUDA events."""
    peak, _ = hbm_peak()
    res = {}
    n = max(5, min(args.steps, 50))
    # The calls that read their input twice (a per-call abs-max pass, then the
    # producer) are timed with L2 flushed to clean lines between calls: timed back
    # to back on the same input, a pass could find the previous call's last reads
    # still in L2, which a caller with new input each call never does.
    l2_scrub = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev)
    l2_clean = torch.ones(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)

    def l2_flush():
        l2_scrub.fill_(1)
        l2_clean.sum()

    def entry(nbytes, per, rows):
        # A launch's CUDA-event time is read in steps of about 1 us on this GPU, so the
        # median of a launch of a few tens of us snaps to a step (28.67 us for anything
        # from 27.6 to 28.7). Launches under 0.1 ms are taken by the mean of their
        # per-launch times instead (each starts at a random phase of the step, so the
        # mean is unbiased); the median is reported beside it.
        med = sorted(per)[len(per) // 2]
        ms = med if med >= 0.1 else sum(per) / len(per)
        gbs = nbytes / (ms * 1e-3) / 1e9
        out = {"gbs": round(gbs, 1), "frac_of_peak": round(gbs / peak, 4),
               "median_launch_ms": round(med, 5), "rows_per_s": round(rows / (ms * 1e-3)),
               "algorithmic_bytes": nbytes, "launches": len(per)}
        if ms != med:
            out["mean_launch_ms"] = round(ms, 5)
            out["timed_by"] = "mean of per-launch times (event steps of about 1 us)"
        return out

    # Each producer's inputs come from fresh device allocations (the caching
    # allocator's blocks released first): the placement of a large strided tensor
    # inside a reused segment can move a launch's time by several per cent.
    # SwiGLU 65,280 x 18,944 (5.6 GB per call: larger than L2)
    torch.cuda.empty_cache()
    gate, up = workloads.swiglu_inputs(dev)
    g = torch.tensor([calibrate_swiglu_gsf(gate, up)], dtype=torch.float32, device=dev)
    c, s = h3q.h3q_swiglu_nvfp4(gate, up, g, stream=stream)
    for _ in range(3):
        h3q.h3q_swiglu_nvfp4(gate, up, g, c, s, stream=stream)
    _, per = time_launches(lambda: h3q.h3q_swiglu_nvfp4(gate, up, g, c, s, stream=stream), n, stream)
    res["swiglu_65280x18944"] = entry(swiglu_bytes(*gate.shape), per, gate.shape[0])
    ipe = recorded_value("swiglu_ring_kernel", os.path.join(ROOT, "profiles", "inst_per_element.txt"))
    if ipe is not None:
        # the instruction-issue bound: every SM sub-partition issuing one warp
        # instruction per cycle at the clock seen under load
        props = torch.cuda.get_device_properties(dev)
        lanes_per_s = props.multi_processor_count * 4 * 32 * args.sm_mhz_seen * 1e6
        ms_issue = gate.numel() * ipe / lanes_per_s * 1e3
        res["swiglu_65280x18944"]["issue_ceiling"] = {
            "thread_inst_per_elem": ipe, "ms_at_full_issue": round(ms_issue, 4),
            "gbs_at_full_issue": round(swiglu_bytes(*gate.shape) / (ms_issue * 1e-3) / 1e9, 1),
            "sm_mhz": args.sm_mhz_seen,
            "source": "ncu smsp__sass_thread_inst_executed.sum per element, profiles/inst_per_element.txt"}
    # dynamic SwiGLU step: abs-max pass, device global scale, producer
    amax_s = torch.zeros(1, dtype=torch.float32, device=dev)
    g_s = torch.empty(1, dtype=torch.float32, device=dev)

    def swiglu_dynamic_step():
        amax_s.zero_()
        h3q.h3q_swiglu_amax(gate, up, amax=amax_s, stream=stream)
        h3q.h3q_global_scale_from_amax(amax_s, g_s, stream=stream)
        h3q.h3q_swiglu_nvfp4(gate, up, g_s, c, s, stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(3):
            swiglu_dynamic_step()
    _, per = time_launches(swiglu_dynamic_step, n, stream, flush=l2_flush)
    sd = entry(swiglu_bytes(*gate.shape), per, gate.shape[0])
    sd["l2"] = "flushed to clean lines between calls"
    sd["two_pass_algorithmic_bytes"] = swiglu_bytes(*gate.shape) + 4 * gate.numel()
    sd["frac_of_peak_two_pass"] = round(sd["two_pass_algorithmic_bytes"] / (sd["median_launch_ms"] * 1e-3) / 1e9
                                        / peak, 4)
    sd["note"] = "abs-max pass + device scale + producer; gate and up read twice, GB/s by the single-pass bytes"
    res["swiglu_dynamic_scale_65280x18944"] = sd
    del c, s, amax_s, g_s

    # SwiGLU of the value-first packed projection with its bias, 65,280 x 2 x 18,944
    del gate, up
    torch.cuda.empty_cache()
    o, bias = workloads.swiglu_packed_inputs(dev)
    c, s = h3q.h3q_swiglu_packed_nvfp4(o, g, bias=bias, stream=stream)
    for _ in range(3):
        h3q.h3q_swiglu_packed_nvfp4(o, g, bias=bias, codes=c, scales=s, stream=stream)
    _, per = time_launches(lambda: h3q.h3q_swiglu_packed_nvfp4(o, g, bias=bias, codes=c, scales=s,
                                                               stream=stream), n, stream)
    res["swiglu_packed_bias_65280x18944"] = entry(swiglu_bytes(ROWS, workloads.FFN) + 4 * workloads.FFN,
                                                  per, ROWS)
    del o, bias, c, s

    # attention-output quantize: 65,280 and 300,000 tokens of 56 x 128
    for tokens in (65280, 300000):
        torch.cuda.empty_cache()
        x = workloads.attention_output(dev, tokens=tokens)
        g = torch.tensor([2688.0 / float(x.abs().max().float())], dtype=torch.float32, device=dev)
        c, s = h3q.h3q_quantize_nvfp4(x, g, stream=stream)
        for _ in range(3):
            h3q.h3q_quantize_nvfp4(x, g, c, s, stream=stream)
        _, per = time_launches(lambda: h3q.h3q_quantize_nvfp4(x, g, c, s, stream=stream), n, stream)
        res[f"attn_out_quantize_{tokens}x7168"] = entry(quantize_bytes(*x.shape), per, tokens)
        if tokens == 65280:
            # the dynamic-scale quantize without caller scratch (abs-max pass, scale, quantize)
            gd = torch.empty(1, dtype=torch.float32, device=dev)
            for _ in range(3):
                h3q.h3q_quantize_nvfp4_dynamic(x, gd, c, s, stream=stream)
            _, per = time_launches(lambda: h3q.h3q_quantize_nvfp4_dynamic(x, gd, c, s, stream=stream), n,
                                   stream, flush=l2_flush)
            dq = entry(quantize_bytes(*x.shape), per, tokens)
            dq["l2"] = "flushed to clean lines between calls"
            dq["two_pass_algorithmic_bytes"] = quantize_bytes(*x.shape) + 2 * x.numel()
            dq["frac_of_peak_two_pass"] = round(dq["two_pass_algorithmic_bytes"] / (dq["median_launch_ms"] * 1e-3)
                                                / 1e9 / peak, 4)
            dq["note"] = ("abs-max pass, then the quantize forming the scale from its partial maxima (a "
                          "programmatic dependent launch), in one call; GB/s by the single-pass bytes")
            res["attn_out_quantize_dynamic_65280x7168"] = dq
            # the checking-path dequantize of that output: codes + scales in, fp32 out
            out = torch.empty(x.shape, dtype=torch.float32, device=dev)
            for _ in range(3):
                h3q.h3q_dequantize_nvfp4(c, s, g, out=out, stream=stream)
            _, per = time_launches(lambda: h3q.h3q_dequantize_nvfp4(c, s, g, out=out, stream=stream), n, stream)
            res["dequantize_65280x7168"] = entry(x.numel() // 2 + padded(tokens) * COLS // 16 + 4 * x.numel() + 4,
                                                 per, tokens)
            del out, gd
        del x, c, s

    # dynamic AdaLN: per-call abs-max pass, device global scale, producer (three
    # launches and an fp32 zero fill per step, no host synchronisation); GB/s by the
    # single-pass algorithmic bytes, although x is read twice
    torch.cuda.empty_cache()
    w = workloads.adaln_inputs(dev)
    amax = torch.zeros(1, dtype=torch.float32, device=dev)
    g = torch.empty(1, dtype=torch.float32, device=dev)
    c = torch.empty((ROWS, COLS // 2), dtype=torch.uint8, device=dev)
    s = torch.empty((padded(ROWS), COLS // 16), dtype=torch.uint8, device=dev)

    rstd = torch.empty(ROWS, dtype=torch.float32, device=dev)

    def dynamic_step():
        # the abs-max pass hands each row's rstd to the second pass, which then
        # forms no statistics of its own
        amax.zero_()
        h3q.h3q_rmsnorm_adaln_amax(w["x"], w["gamma"], w["table"], rows_per_frame=RPF, eps=w["eps"],
                                   amax=amax, row_rstd=rstd, stream=stream)
        h3q.h3q_global_scale_from_amax(amax, g, stream=stream)
        h3q.h3q_rmsnorm_adaln_nvfp4_from_rstd(w["x"], w["gamma"], w["table"], rstd, g, rows_per_frame=RPF,
                                              codes=c, scales=s, stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(3):
            dynamic_step()
    _, per = time_launches(dynamic_step, n, stream, flush=l2_flush)
    res["adaln_dynamic_scale_65280x7168"] = entry(adaln_bytes(ROWS, COLS, FRAMES), per, ROWS)
    res["adaln_dynamic_scale_65280x7168"]["l2"] = "flushed to clean lines between calls"
    res["adaln_dynamic_scale_65280x7168"]["note"] = ("abs-max pass (writing each row's rstd) + device scale + "
                                                     "producer taking the rstd; x is read twice, GB/s by the "
                                                     "single-pass bytes")
    # the least a per-call abs-max scale can move: x read by both passes (the whole
    # tensor's maximum is needed before any row is quantized), the outputs once
    two_pass = adaln_bytes(ROWS, COLS, FRAMES) + 2 * ROWS * COLS + 2 * COLS + FRAMES * 2 * COLS * 2 + 2 * 4 * ROWS
    dyn = res["adaln_dynamic_scale_65280x7168"]
    dyn["two_pass_algorithmic_bytes"] = two_pass
    dyn["frac_of_peak_two_pass"] = round(two_pass / (dyn["median_launch_ms"] * 1e-3) / 1e9 / peak, 4)
    del w, c, s, rstd

    # residual fold + RMSNorm + AdaLN: h (fp32) is read and written back each launch
    torch.cuda.empty_cache()
    w = workloads.residual_inputs(dev)
    g = torch.tensor([90.0], dtype=torch.float32, device=dev)
    c = torch.empty((ROWS, COLS // 2), dtype=torch.uint8, device=dev)
    s = torch.empty((padded(ROWS), COLS // 16), dtype=torch.uint8, device=dev)

    def residual_step():
        h3q.h3q_residual_rmsnorm_adaln_nvfp4(w["h"], w["o"], w["gate"], w["gamma"], w["table"], g,
                                             bias=w["bias"], rows_per_frame=RPF, eps=w["eps"],
                                             codes=c, scales=s, stream=stream)

    for _ in range(3):
        residual_step()
    _, per = time_launches(residual_step, n, stream)
    res["residual_adaln_65280x7168"] = entry(residual_bytes(ROWS, COLS, FRAMES), per, ROWS)
    del w, c, s

    # QKV epilogue: 65,280 tokens x 56 heads x 128 (ROT 64), q, k, v column slices of
    # one packed projection, bf16 [rows, heads, 128] outputs
    torch.cuda.empty_cache()
    w = workloads.qkv_inputs(dev)
    outs = h3q.h3q_qkv_epilogue(w["q"], w["k"], w["v"], w["biases"], w["cos"], w["sin"], w["heads"],
                                w["eps"], stream=stream)

    def qkv_step():
        h3q.h3q_qkv_epilogue(w["q"], w["k"], w["v"], w["biases"], w["cos"], w["sin"], w["heads"],
                             w["eps"], outs=outs, stream=stream)

    for _ in range(3):
        qkv_step()
    _, per = time_launches(qkv_step, n, stream)
    res["qkv_epilogue_65280x56x128_rot64"] = entry(qkv_bytes(ROWS, w["heads"], w["head_dim"], w["rot"]),
                                                   per, ROWS)
    del w, outs

    # standalone quantize 8,192 x 7,168 (150 MB: near L2, so L2 is flushed before each launch)
    torch.cuda.empty_cache()
    x = workloads.quantize_inputs(dev)
    g = torch.tensor([2688.0 / float(x.float().abs().max())], dtype=torch.float32, device=dev)
    c, s = h3q.h3q_quantize_nvfp4(x, g, stream=stream)
    _, per = time_launches(lambda: h3q.h3q_quantize_nvfp4(x, g, c, s, stream=stream), n, stream,
                           flush=lambda: l2_scrub.fill_(1))
    res["quantize_8192x7168_l2_flushed"] = entry(quantize_bytes(*x.shape), per, 8192)
    # The write leaves L2 full of dirty lines, whose write-back then falls inside the timed launch.
    # Reading a second 2 x L2 buffer after it (l2_flush) writes them back first: the launch starts
    # on an L2 of clean lines that hold none of its inputs.
    _, per = time_launches(lambda: h3q.h3q_quantize_nvfp4(x, g, c, s, stream=stream), n, stream,
                           flush=l2_flush)
    res["quantize_8192x7168_l2_flushed_clean"] = entry(quantize_bytes(*x.shape), per, 8192)
    del x, c, s

    # The FFN-up projection as a block-scaled NVFP4 GEMM with the SwiGLU + NVFP4
    # epilogue (65,280 x 7,168 -> 2 x 18,944): tensor-bound, so TFLOP/s against the
    # NVFP4 dense peak.
    torch.cuda.empty_cache()
    ops, flops = gemm_operands(h3q, dev, stream, ROWS)
    c, s = h3q.h3q_gemm_swiglu_nvfp4(*ops, stream=stream)
    for _ in range(3):
        h3q.h3q_gemm_swiglu_nvfp4(*ops, c, s, stream=stream)
    _, per = time_launches(lambda: h3q.h3q_gemm_swiglu_nvfp4(*ops, c, s, stream=stream), min(n, 20), stream)
    ms = sorted(per)[len(per) // 2]
    tpeak, tsrc = fp4_peak()
    tflops = flops / (ms * 1e-3) / 1e12
    res["gemm_swiglu_nvfp4_65280x7168x37888"] = {
        "bound": "tensor", "tflops": round(tflops, 1), "peak_tflops": round(tpeak, 1), "peak_source": tsrc,
        "frac_of_peak": round(tflops / tpeak, 4), "frac_of_nominal_13_5_pf": round(tflops / 13500.0, 4),
        "median_launch_ms": round(ms, 4), "flops": flops, "rows_per_s": round(ROWS / (ms * 1e-3)),
        "launches": len(per), "error_flag": h3q.h3q_kernel_error_flag()}
    del ops, c, s
    torch.cuda.empty_cache()

    # The small cases, each launch after the same clean-lines flush. A launch's fixed cost is most of
    # their time, so they measure latency, not bandwidth.
    #  - the tiny AdaLN case (64 x 256);
    #  - the ragged attention-output quantize at 1,000 tokens (18 MB).
    w = workloads.tiny_adaln_inputs(dev)
    g = torch.tensor([calibrate_adaln_gsf(w)], dtype=torch.float32, device=dev)
    c, s = h3q.h3q_rmsnorm_adaln_nvfp4(w["x"], w["gamma"], w["table"], g, rows_per_frame=w["rows_per_frame"],
                                       eps=w["eps"], stream=stream)
    _, per = time_launches(lambda: h3q.h3q_rmsnorm_adaln_nvfp4(
        w["x"], w["gamma"], w["table"], g, rows_per_frame=w["rows_per_frame"], eps=w["eps"], codes=c,
        scales=s, stream=stream), n, stream, flush=l2_flush)
    res["adaln_tiny_64x256_l2_flushed_clean"] = entry(adaln_bytes(64, 256, w["table"].shape[0]), per, 64)
    x = workloads.attention_output(dev, tokens=1000)
    g = torch.tensor([2688.0 / float(x.abs().max().float())], dtype=torch.float32, device=dev)
    c, s = h3q.h3q_quantize_nvfp4(x, g, stream=stream)
    _, per = time_launches(lambda: h3q.h3q_quantize_nvfp4(x, g, c, s, stream=stream), n, stream, flush=l2_flush)
    res["attn_out_quantize_1000x7168_l2_flushed_clean"] = entry(quantize_bytes(*x.shape), per, 1000)
    del w, x, c, s, l2_scrub, l2_clean
    torch.cuda.empty_cache()
    if not args.no_cpu_baseline:
        for key, kind in (("swiglu_65280x18944", "swiglu"), ("swiglu_packed_bias_65280x18944", "swiglu_packed"),
                          ("attn_out_quantize_65280x7168", "quantize"), ("residual_adaln_65280x7168", "residual"),
                          ("qkv_epilogue_65280x56x128_rot64", "qkv")):
            res[key]["cpu_oracle"] = producer_oracle(kind)
    return res


# --------------------------------------------------------------------------- #
# CPU oracle (cpu_baseline and --impl reference)                                #
# --------------------------------------------------------------------------- #

def _oracle_adaln_sample(rows: int, seed: int):
    import numpy as np

    w = workloads.adaln_inputs("cpu", rows=rows, seed=seed)
    bits = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)  # noqa: E731
    frames = (np.arange(rows) + seed * rows) // RPF % FRAMES
    return bits(w["x"]), bits(w["gamma"]), bits(w["table"]), frames, w["eps"]


def cpu_baseline(seconds: float = 15.0, rows_per_chunk: int = 255):
    """The oracle as it stands on the host cores, over chunks of the AdaLN workload
    until about `seconds` of work has run; GB/s from the same algorithmic bytes."""
    import oracle

    threads = os.cpu_count() or 1
    oracle.lib()
    done_rows, spent, chunk = 0, 0.0, 0
    while spent < seconds:
        x, gm, tb, fr, eps = _oracle_adaln_sample(rows_per_chunk, seed=100 + chunk)
        t0 = time.perf_counter()
        oracle.adaln_rows(x, gm, tb, fr, eps, 1.0, threads=threads)
        spent += time.perf_counter() - t0
        done_rows += rows_per_chunk
        chunk += 1
    nbytes = done_rows / ROWS * adaln_bytes(ROWS, COLS, FRAMES)
    # the same oracle on one core, over a shorter sample
    one_rows, one_spent, one_chunk = 0, 0.0, 0
    while one_spent < max(1.0, seconds / 5):
        x, gm, tb, fr, eps = _oracle_adaln_sample(rows_per_chunk, seed=500 + one_chunk)
        t0 = time.perf_counter()
        oracle.adaln_rows(x, gm, tb, fr, eps, 1.0, threads=1)
        one_spent += time.perf_counter() - t0
        one_rows += rows_per_chunk
        one_chunk += 1
    one_bytes = one_rows / ROWS * adaln_bytes(ROWS, COLS, FRAMES)
    return {"value": round(nbytes / spent / 1e9, 4), "unit": "GB/s", "cores": threads,
            "kind": "oracle",
            "sample": f"{done_rows} rows x {COLS} of the AdaLN workload ({chunk} chunks of "
                      f"{rows_per_chunk} rows, {spent:.1f} s on {threads} threads); GB/s by the "
                      "same algorithmic-byte count as the GPU line",
            "single_core": {"value": round(one_bytes / one_spent / 1e9, 4), "unit": "GB/s", "cores": 1,
                            "sample": f"{one_rows} rows x {COLS} ({one_spent:.1f} s on one thread)"}}


def producer_oracle(kind: str, seconds: float = 2.0, rows: int = 64) -> dict:
    """One producer's oracle as it stands on the host cores, over chunks of `rows`
    rows of its workload until about `seconds` of work has run; GB/s by the same
    algorithmic bytes per row as the GPU entry."""
    import numpy as np
    import oracle

    threads = os.cpu_count() or 1
    bits = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)  # noqa: E731
    F = workloads.FFN
    done, spent, chunk = 0, 0.0, 0
    while spent < seconds:
        seed = 300 + chunk
        if kind == "swiglu":
            gate, up = workloads.swiglu_inputs("cpu", rows=rows, seed=seed)
            args_, fn = (bits(gate), bits(up), 1.0), oracle.swiglu_rows
            per_row = swiglu_bytes(ROWS, F) / ROWS
        elif kind == "swiglu_packed":
            o, b = workloads.swiglu_packed_inputs("cpu", rows=rows, seed=seed)
            args_, fn = (bits(o), bits(b), 1.0), oracle.swiglu_packed_rows
            per_row = (swiglu_bytes(ROWS, F) + 4 * F) / ROWS
        elif kind == "quantize":
            x = workloads.attention_output("cpu", tokens=rows, seed=seed)
            args_, fn = (bits(x), 1.0), oracle.quantize_rows
            per_row = quantize_bytes(ROWS, COLS) / ROWS
        elif kind == "residual":
            w = workloads.residual_inputs("cpu", rows=rows, frames=1, seed=seed)
            fr = np.zeros(rows, np.int64)
            args_ = (w["h"].numpy(), bits(w["o"]), bits(w["bias"]), bits(w["gate"]), bits(w["gamma"]),
                     bits(w["table"]), fr, w["eps"], 1.0)
            fn = oracle.residual_adaln_rows
            per_row = residual_bytes(ROWS, COLS, FRAMES) / ROWS
        elif kind == "qkv":
            w = workloads.qkv_inputs("cpu", rows=rows, seed=seed)
            per_row = qkv_bytes(ROWS, w["heads"], w["head_dim"], w["rot"]) / ROWS
            t0 = time.perf_counter()
            for i, name in enumerate("qkv"):
                oracle.qkv_epilogue_rows(bits(w[name]), bits(w["biases"][i]), w["heads"], bits(w["cos"]),
                                         bits(w["sin"]), w["eps"], is_v=(name == "v"), threads=threads)
            spent += time.perf_counter() - t0
            done += rows
            chunk += 1
            continue
        else:
            raise ValueError(kind)
        t0 = time.perf_counter()
        fn(*args_, threads=threads)
        spent += time.perf_counter() - t0
        done += rows
        chunk += 1
    return {"gbs": round(done * per_row / spent / 1e9, 4), "cores": threads, "kind": "oracle",
            "sample": f"{done} rows in {chunk} chunks of {rows}, {spent:.1f} s on {threads} threads"}


def run_reference(args, rank, world):
    """The CPU oracle timed on the host cores: each step is a bounded sample of the
    AdaLN workload (rows_per_step rows), after `warmup` untimed steps."""
    import oracle

    if rank != 0:
        return None
    threads = os.cpu_count() or 1
    oracle.lib()
    rows_per_step = args.reference_rows
    spent = 0.0
    for i in range(args.warmup + args.steps):
        x, gm, tb, fr, eps = _oracle_adaln_sample(rows_per_step, seed=200 + i)
        t0 = time.perf_counter()
        oracle.adaln_rows(x, gm, tb, fr, eps, 1.0, threads=threads)
        if i >= args.warmup:
            spent += time.perf_counter() - t0
    nbytes = rows_per_step / ROWS * adaln_bytes(ROWS, COLS, FRAMES) * args.steps
    value = round(nbytes / spent / 1e9, 4)
    sample = (f"each step {rows_per_step} rows x {COLS} of the AdaLN workload (a bounded sample of its "
              f"{ROWS} rows), {threads} threads; GB/s by the same algorithmic-byte count as the GPU line")
    return {
        "impl": "reference",
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(spent / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {**workload_config(), "parallelism": "host cores"},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


# --------------------------------------------------------------------------- #
# one producer alone (profiling captures and sweeps)                            #
# --------------------------------------------------------------------------- #

def run_single(args, dev):
    """W warm-up and K timed launches of one producer at --rows rows (cols as in the
    workloads); prints one JSON line.  Used for ncu captures of a small case."""
    import nvfp4_activation_quantize_gb300 as h3q

    stream = torch.cuda.current_stream(dev)
    kind = args.kernel
    if kind == "adaln":
        rows = args.rows or ROWS
        w = workloads.adaln_inputs(dev, rows=rows, frames=max(1, -(-rows // RPF)))
        g = torch.tensor([calibrate_adaln_gsf(w)], dtype=torch.float32, device=dev)
        c = torch.empty((rows, COLS // 2), dtype=torch.uint8, device=dev)
        s = torch.empty((padded(rows), COLS // 16), dtype=torch.uint8, device=dev)
        fn = lambda: h3q.h3q_rmsnorm_adaln_nvfp4(  # noqa: E731
            w["x"], w["gamma"], w["table"], g, rows_per_frame=RPF, eps=w["eps"], codes=c, scales=s,
            stream=stream)
        nbytes = adaln_bytes(rows, COLS, w["table"].shape[0])
    elif kind == "swiglu":
        rows = args.rows or ROWS
        gate, up = workloads.swiglu_inputs(dev, rows=rows)
        g = torch.tensor([calibrate_swiglu_gsf(gate, up)], dtype=torch.float32, device=dev)
        c, s = h3q.h3q_swiglu_nvfp4(gate, up, g, stream=stream)
        fn = lambda: h3q.h3q_swiglu_nvfp4(gate, up, g, c, s, stream=stream)  # noqa: E731
        nbytes = swiglu_bytes(rows, workloads.FFN)
    elif kind == "swiglu_packed":
        rows = args.rows or ROWS
        o, bias = workloads.swiglu_packed_inputs(dev, rows=rows)
        f = workloads.FFN
        g = torch.tensor([calibrate_swiglu_gsf(o[:, f:], o[:, :f])], dtype=torch.float32, device=dev)
        c, s = h3q.h3q_swiglu_packed_nvfp4(o, g, bias=bias, stream=stream)
        fn = lambda: h3q.h3q_swiglu_packed_nvfp4(o, g, bias=bias, codes=c, scales=s,  # noqa: E731
                                                 stream=stream)
        nbytes = swiglu_bytes(rows, workloads.FFN) + 4 * workloads.FFN
    elif kind == "residual":
        rows = args.rows or ROWS
        w = workloads.residual_inputs(dev, rows=rows, frames=max(1, -(-rows // RPF)))
        g = torch.tensor([90.0], dtype=torch.float32, device=dev)
        c = torch.empty((rows, COLS // 2), dtype=torch.uint8, device=dev)
        s = torch.empty((padded(rows), COLS // 16), dtype=torch.uint8, device=dev)
        fn = lambda: h3q.h3q_residual_rmsnorm_adaln_nvfp4(  # noqa: E731
            w["h"], w["o"], w["gate"], w["gamma"], w["table"], g, bias=w["bias"], rows_per_frame=RPF,
            eps=w["eps"], codes=c, scales=s, stream=stream)
        nbytes = residual_bytes(rows, COLS, w["table"].shape[0])
    elif kind == "quantize_dynamic":
        rows = args.rows or ROWS
        x = workloads.attention_output(dev, tokens=rows)
        c, s, g = h3q.h3q_quantize_nvfp4_dynamic(x, stream=stream)
        fn = lambda: h3q.h3q_quantize_nvfp4_dynamic(x, global_scale=g, codes=c, scales=s,  # noqa: E731
                                                    stream=stream)
        nbytes = quantize_bytes(rows, COLS)  # by the single-pass bytes (x is read twice)
    elif kind == "dequantize":
        rows = args.rows or ROWS
        x = workloads.attention_output(dev, tokens=rows)
        g = torch.tensor([2688.0 / float(x.abs().max().float())], dtype=torch.float32, device=dev)
        c, s = h3q.h3q_quantize_nvfp4(x, g, stream=stream)
        out = torch.empty(x.shape, dtype=torch.float32, device=dev)
        fn = lambda: h3q.h3q_dequantize_nvfp4(c, s, g, out=out, stream=stream)  # noqa: E731
        nbytes = rows * COLS // 2 + padded(rows) * COLS // 16 + 4 * rows * COLS + 4
    elif kind == "qkv":
        rows = args.rows or ROWS
        w = workloads.qkv_inputs(dev, rows=rows)
        outs = h3q.h3q_qkv_epilogue(w["q"], w["k"], w["v"], w["biases"], w["cos"], w["sin"],
                                    w["heads"], w["eps"], stream=stream)
        fn = lambda: h3q.h3q_qkv_epilogue(  # noqa: E731
            w["q"], w["k"], w["v"], w["biases"], w["cos"], w["sin"], w["heads"], w["eps"], outs=outs,
            stream=stream)
        nbytes = qkv_bytes(rows, w["heads"], w["head_dim"], w["rot"])
    elif kind == "gemm":
        rows = args.rows or ROWS
        ops, flops = gemm_operands(h3q, dev, stream, rows)
        c, s = h3q.h3q_gemm_swiglu_nvfp4(*ops, stream=stream)
        fn = lambda: h3q.h3q_gemm_swiglu_nvfp4(*ops, c, s, stream=stream)  # noqa: E731
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        _, per = time_launches(fn, args.steps, stream)
        ms = sorted(per)[len(per) // 2]
        tpeak, tsrc = fp4_peak()
        tflops = flops / (ms * 1e-3) / 1e12
        return {"kernel": kind, "rows": rows, "median_launch_ms": round(ms, 4), "tflops": round(tflops, 1),
                "frac_of_peak": round(tflops / tpeak, 4), "peak_tflops": round(tpeak, 1), "peak_source": tsrc,
                "flops": flops, "launches": args.steps, "warmup": args.warmup,
                "error_flag": h3q.h3q_kernel_error_flag()}
    else:
        rows = args.rows or ROWS
        x = workloads.attention_output(dev, tokens=rows)
        g = torch.tensor([2688.0 / float(x.abs().max().float())], dtype=torch.float32, device=dev)
        c, s = h3q.h3q_quantize_nvfp4(x, g, stream=stream)
        fn = lambda: h3q.h3q_quantize_nvfp4(x, g, c, s, stream=stream)  # noqa: E731
        nbytes = quantize_bytes(rows, COLS)
    for _ in range(args.warmup):
        fn()
    torch.cuda.synchronize()
    _, per = time_launches(fn, args.steps, stream)
    ms = sorted(per)[len(per) // 2]
    peak, _ = hbm_peak()
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"kernel": kind, "rows": rows, "median_launch_ms": round(ms, 5), "gbs": round(gbs, 1),
            "frac_of_peak": round(gbs / peak, 4), "algorithmic_bytes": nbytes,
            "launches": args.steps, "warmup": args.warmup}


# --------------------------------------------------------------------------- #

def main(argv=None):
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--soak", type=float, default=1.0, help="untimed seconds of steps before timing")
    p.add_argument("--cpu-seconds", type=float, default=15.0)
    p.add_argument("--reference-rows", type=int, default=510)
    p.add_argument("--no-extras", action="store_true", help="skip producers, e2e and cpu baseline")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--kernel", choices=["adaln", "swiglu", "swiglu_packed", "quantize", "quantize_dynamic",
                                        "residual", "qkv", "dequantize", "gemm"],
                   help="time one producer alone (for profiling); prints a short JSON line")
    p.add_argument("--rows", type=int, default=0, help="rows for --kernel (default: full size)")
    args = p.parse_args(argv)
    if args.warmup < 3:
        p.error("--warmup must be at least 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        res = run_reference(args, rank, world)
        if res is not None:
            print(json.dumps(res), flush=True)
        return 0

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (there is no CPU path)")
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    if args.kernel:
        print(json.dumps(run_single(args, dev)), flush=True)
        return 0
    if world > 1:
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        torch.distributed.init_process_group("nccl", device_id=dev)
    try:
        res = run_ours(args, rank, world, dev)
    finally:
        if world > 1:
            torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(res), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
