#!/usr/bin/env python
"""Benchmark of the MoE FFN forward pass (libmoe, C ABI) on B300 GPUs.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

One step = one moe_forward over one batch of T tokens of the workload (route, dispatch,
grouped SwiGLU experts, shared experts, combine), inputs resident in HBM, L2 flushed (256 MiB
write) between steps, each step timed with CUDA events on the launching stream.  W warm-up
steps, a 0.25 s pause while the clock samplers start, then K timed steps back to back.  The stage
split comes from a second pass of moe_forward_profiled (the same kernels with events at the
stage boundaries, which keep each kernel from starting during its predecessor's tail).  With N > 1 (torchrun, one
rank per GPU) every rank runs its own batch with replicated weights (the layer is per-token,
so tokens shard with no exchange): weak scaling, no collective on the data path.

Rank 0 prints one JSON line.  `value` = tokens of all ranks / max-over-ranks device time.
`e2e` is the same through moe_forward_host_async with x and y in pinned host memory (two
streams, so that one step's host copies overlap another step's kernels); `e2e.sync` is the
synchronous moe_forward_host, step after step.  `roofline` is the W1/W2 + SwiGLU grouped GEMM
(the dominant kernel).  `cpu_baseline` is the CPU oracle on a bounded sample on this host.
At N = 1 the line also carries `workloads`: the same record (tokens/s, stage times, expert-GEMM
fraction of the bf16 peak, roofline, e2e, its own CPU-oracle sample) for the Hunyuan-A13B-shaped,
DeepSeek-V3-shaped and float32 workloads.  `--impl reference` times the oracle alone.
"""
from __future__ import annotations

import argparse
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

import workloads as wl  # noqa: E402

METRIC = "MoE-layer tokens/sec on 1 B300; expert-GEMM % of bf16 peak; decode HBM GB/s"
DEFAULT_WORKLOAD = "mixtral_prefill"
DECODE_WORKLOAD = "mixtral_decode"
# measured after the headline workload in the default run (N = 1): the Hunyuan-A13B-shaped and
# DeepSeek-V3-shaped prefill layers and the float32 correctness layer
EXTRA_WORKLOADS = ("hunyuan_a13b", "deepseek_v3", "tiny_f32")
# tokens per CPU-oracle sample, sized for a few seconds of host time per workload
ORACLE_SAMPLE_TOKENS = {"tiny_f32": 64, "mixtral_prefill": 64, "mixtral_decode": 16, "hunyuan_a13b": 32,
                        "deepseek_v3": 8}
FLUSH_BYTES = 256 << 20

# DRAM bytes (read + write) per launch of each workload's W1/W2 SwiGLU GEMM, from one-pass ncu
# captures (profiles/): the Mixtral- and Hunyuan-shaped launches at full size, the
# DeepSeek-V3-shaped one on 32 of 256 experts and 1024 of 8192 tokens, x 8.  Valid only for the
# kernel code it was taken on (gemm_tc.cu without comments, by sha256); null otherwise.
NCU_TRAFFIC = {"code_sha256": "2574ae6fc36a18dfad5270e6d08b0198df80815f728dbaa1555858fd5f72a499",
               "bytes_per_launch": {"mixtral_prefill": 2181.8e6, "hunyuan_a13b": 4272.5e6, "deepseek_v3": 16470.4e6}}


def _code_sha256(path):
    """sha256 of a C++/CUDA source with its // comments and blank lines removed: the traffic
    figure belongs to the code, and stays valid across comment edits."""
    import re
    lines = []
    for line in open(path).read().splitlines():
        line = re.sub(r"//.*$", "", line).rstrip()
        if line:
            lines.append(line)
    return hashlib.sha256("\n".join(lines).encode()).hexdigest()


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0, "source": "fallback"}


# ----------------------------------------------------------------------------- clocks

IDLE_BEFORE_TIMED_S = 0.25


class ClockSampler:
    """SM clock and clock-event reasons while the timed region runs, from two sources: the
    nvidia-smi query line every 200 ms, and NVML in this process every ~2 ms.  A step of a few
    milliseconds makes a timed region shorter than nvidia-smi's interval, so most of its samples
    fall before and after the region (on an idle, fully clocked GPU); the summary takes the NVML
    samples between mark_start() and mark_end() when there are enough of them."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,utilization.gpu,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    # NVML clock-event reason bits (nvmlClocksEventReason*)
    NVML_REASONS = ((0x4, "sw_power_cap"), (0x8, "hw_slowdown"), (0x20, "sw_thermal_slowdown"),
                    (0x40, "hw_thermal_slowdown"), (0x80, "hw_power_brake_slowdown"))

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.lines = []
        self.nvml = []          # (host time, sm MHz, reason bits)
        self.nvml_max = None
        self.nvml_error = None
        self.region = None
        self._stop = threading.Event()
        self._nvml_thread = None

    def _device_id(self):
        """The GPU as nvidia-smi and NVML name it: its UUID (CUDA and NVML number GPUs
        differently when CUDA_VISIBLE_DEVICES is set), else the CUDA index."""
        try:
            import torch
            u = str(torch.cuda.get_device_properties(self.dev).uuid)
            return u if u.startswith("GPU-") else "GPU-" + u
        except Exception:
            return str(self.dev)

    @staticmethod
    def _nvml_api():
        """The NVML queries the sampler needs, through the driver's libnvidia-ml (its public
        C API, called with ctypes), else through the pynvml package."""
        import ctypes
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
        except OSError:
            lib = None
        if lib is not None:
            dev_t = ctypes.c_void_p

            def check(r, what):
                if r != 0:
                    raise RuntimeError("%s returned %d" % (what, r))
            check(lib.nvmlInit_v2(), "nvmlInit_v2")

            def handle(ident, index):
                h = dev_t()
                if lib.nvmlDeviceGetHandleByUUID(ident.encode(), ctypes.byref(h)) != 0:
                    check(lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index), ctypes.byref(h)),
                          "nvmlDeviceGetHandleByIndex_v2")
                return h

            def uint_query(fn, h, *args):
                v = ctypes.c_uint()
                check(fn(h, *args, ctypes.byref(v)), fn.__name__)
                return v.value

            def reasons(h):
                v = ctypes.c_ulonglong()
                check(lib.nvmlDeviceGetCurrentClocksEventReasons(h, ctypes.byref(v)), "reasons")
                return v.value
            return {"handle": handle,
                    "sm": lambda h: uint_query(lib.nvmlDeviceGetClockInfo, h, ctypes.c_int(1)),
                    "sm_max": lambda h: uint_query(lib.nvmlDeviceGetMaxClockInfo, h, ctypes.c_int(1)),
                    "reasons": reasons,
                    "shutdown": lib.nvmlShutdown}
        import pynvml as nv
        nv.nvmlInit()

        def handle(ident, index):
            try:
                return nv.nvmlDeviceGetHandleByUUID(ident)
            except Exception:
                return nv.nvmlDeviceGetHandleByIndex(index)
        return {"handle": handle,
                "sm": lambda h: nv.nvmlDeviceGetClockInfo(h, nv.NVML_CLOCK_SM),
                "sm_max": lambda h: nv.nvmlDeviceGetMaxClockInfo(h, nv.NVML_CLOCK_SM),
                "reasons": nv.nvmlDeviceGetCurrentClocksEventReasons,
                "shutdown": nv.nvmlShutdown}

    def _nvml_loop(self, ident):
        try:
            api = self._nvml_api()
        except Exception as e:
            self.nvml_error = "init: %s" % e
            return
        try:
            h = api["handle"](ident, self.dev)
            self.nvml_max = float(api["sm_max"](h))
            while not self._stop.is_set():
                t = time.perf_counter()
                self.nvml.append((t, float(api["sm"](h)), int(api["reasons"](h))))
                time.sleep(0.002)
        except Exception as e:
            self.nvml_error = "sampling: %s" % e
        finally:
            try:
                api["shutdown"]()
            except Exception:
                pass

    def __enter__(self):
        ident = self._device_id()
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", ident, "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, ValueError):
            self.proc = None
        self._nvml_thread = threading.Thread(target=self._nvml_loop, args=(ident,), daemon=True)
        self._nvml_thread.start()
        time.sleep(IDLE_BEFORE_TIMED_S)   # both samplers running before the timed region starts
        return self

    def mark_start(self):
        self.region = [time.perf_counter(), None]

    def mark_end(self):
        if self.region:
            self.region[1] = time.perf_counter()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        time.sleep(0.25)
        self._stop.set()
        if self._nvml_thread is not None:
            self._nvml_thread.join(timeout=5)
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def _smi_summary(self):
        rows = []
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 10:
                continue
            try:
                rows.append({"sm": float(f[1]), "max": float(f[2]), "util": float(f[4]),
                             "hw": f[6], "hwt": f[7], "swt": f[8], "pcap": f[9]})
            except ValueError:
                continue
        if not rows:
            return None
        load = [r for r in rows if r["util"] >= 50] or rows
        reasons = set()
        for r in load:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("pcap", "sw_power_cap")):
                if r[key].lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in load), "sm_max_mhz": max(r["max"] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows), "samples_under_load": len(load)}

    def summary(self):
        smi = self._smi_summary()
        inside = []
        if self.region and self.region[1] is not None:
            inside = [r for r in self.nvml if self.region[0] <= r[0] <= self.region[1]]
        if len(inside) >= 3:
            reasons = set(smi["reasons"]) if smi else set()
            for _, _, bits in inside:
                for bit, name in self.NVML_REASONS:
                    if bits & bit:
                        reasons.add(name)
            out = {"sm_mhz": statistics.median(r[1] for r in inside),
                   "sm_mhz_min": min(r[1] for r in inside),
                   "sm_max_mhz": self.nvml_max or (smi["sm_max_mhz"] if smi else None),
                   "reasons": sorted(reasons), "source": "NVML every ~2 ms inside the timed region",
                   "samples": len(inside)}
            if smi:
                out["nvidia_smi"] = smi
            return out
        if smi:
            smi["source"] = "nvidia-smi every 200 ms"
            smi["nvml"] = {"samples": len(self.nvml), "in_region": len(inside), "error": self.nvml_error}
        return smi


# ----------------------------------------------------------------------------- distributed

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(v: float, world: int, device=None) -> float:
    if world <= 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ----------------------------------------------------------------------------- host and CPU oracle legs

def host_cpu():
    """(CPU model name, CPUs this process may run on)."""
    model = None
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.startswith("model name"):
                    model = line.split(":", 1)[1].strip()
                    break
    except OSError:
        pass
    try:
        n = len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        n = os.cpu_count() or 1
    return model, n


def cpu_threads() -> int:
    """Threads of numpy's BLAS pool: the most threads the oracle runs at once (its matrix
    products; the rest of it is single-threaded numpy)."""
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("internal_api") in ("openblas", "mkl")]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count() or 1


def oracle_experts_needed(shape, x_rows, W_g, logit_bias):
    """Experts that the oracle's routing of these token rows picks: only their weights need a
    host copy for the CPU-oracle sample."""
    from oracle import moe_oracle as orc
    r = orc.route(wl.to_f64(x_rows, shape.dtype), wl.to_f64(W_g, shape.dtype), shape.k, shape.scoring, logit_bias)
    # the grouped evaluation also reads expert 0's W3 for the output width
    return sorted(set(int(e) for e in np.unique(r["idx"])) | {0})


def oracle_sample(shape, x_rows, W_g, logit_bias, get_w) -> float:
    """The CPU oracle, as it stands, on the given token rows: router, dispatch, one float64
    SwiGLU per expert block, combine (+ shared experts).  Returns the wall seconds (the inputs
    are drawn beforehand and not timed)."""
    from oracle import moe_oracle as orc
    x64 = wl.to_f64(x_rows, shape.dtype)
    Wg = wl.to_f64(W_g, shape.dtype)
    t0 = time.perf_counter()
    orc.forward(x64, Wg, get_w, shape.E, shape.k, shape.scoring, logit_bias, None, shape.n_shared)
    return time.perf_counter() - t0


def sample_tokens(args, shape) -> int:
    n = args.ref_tokens if args.ref_tokens else ORACLE_SAMPLE_TOKENS.get(shape.name, 16)
    return max(1, min(shape.T, n))


def cpu_record(shape, seconds, n_tok, per="one pass") -> dict:
    model, ncpu = host_cpu()
    return {"value": n_tok / seconds, "unit": "tokens/s", "cores": cpu_threads(), "host_cpus": ncpu,
            "cpu_model": model, "kind": "oracle", "seconds": round(seconds, 3),
            "sample": "first %d of the workload's %d tokens, %s (fp32 router, fp64 experts and combine; "
                      "a correctness oracle, not a tuned CPU MoE)" % (n_tok, shape.T, per)}


def host_weights(shape, experts, seed=0):
    """Host copies (stored dtype) of the routed experts in `experts` and of every shared expert,
    drawn in parallel."""
    from concurrent.futures import ThreadPoolExecutor
    jobs = [(name, e) for name in ("W1", "W2", "W3") for e in experts]
    jobs += [(name, s) for name in (("Ws1", "Ws2", "Ws3") if shape.n_shared else ()) for s in range(shape.n_shared)]
    _, ncpu = host_cpu()
    with ThreadPoolExecutor(max(4, min(32, ncpu))) as ex:
        arrays = list(ex.map(lambda j: wl.gen_expert(shape, j[0], j[1], seed), jobs))
    return dict(zip(jobs, arrays))


def workload_config(shape, world) -> dict:
    return {"workload": shape.name, "T": shape.T, "d": shape.d, "d_ff": shape.d_ff, "E": shape.E, "k": shape.k,
            "scoring": shape.scoring, "n_shared": shape.n_shared, "d_ff_shared": shape.d_ff_shared,
            "logit_bias_std": shape.logit_bias_std, "tokens_per_gpu": shape.T,
            "parallelism": "replicas (token shards)" if world > 1 else "1 GPU",
            "l2": "flushed between steps (256 MiB write)"}


def run_reference(args, shape, world, rank):
    if rank != 0:
        return 0
    n_tok = sample_tokens(args, shape)
    x = wl.gen_x(shape, 0)[:n_tok]
    W_g = wl.gen_router(shape, 0)
    lb = wl.gen_logit_bias(shape, 0)
    host = host_weights(shape, oracle_experts_needed(shape, x, W_g, lb))
    get_w = lambda name, e: wl.to_f64(host[(name, e)], shape.dtype)
    for _ in range(args.warmup):
        oracle_sample(shape, x, W_g, lb, get_w)
    times = [oracle_sample(shape, x, W_g, lb, get_w) for _ in range(args.steps)]
    total = sum(times)
    value = n_tok * args.steps / total
    cpu = cpu_record(shape, total / args.steps, n_tok, "per step")
    cpu["value"] = value
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded generator)", "config": workload_config(shape, world),
            "cpu_baseline": cpu,
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


# ----------------------------------------------------------------------------- GPU leg

def upload_weights(shape, torch, seed=0, keep=()):
    """Draw every expert matrix (in parallel), copy it to the device, and keep host copies of
    the routed experts in `keep` and, when `keep` is not None, of the shared experts."""
    from concurrent.futures import ThreadPoolExecutor
    dt = torch.bfloat16 if shape.dtype == "bf16" else torch.float32
    W = {}
    jobs = []
    for name in ("W1", "W2", "W3") + (("Ws1", "Ws2", "Ws3") if shape.n_shared else ()):
        n = shape.n_shared if name.startswith("Ws") else shape.E
        rows, cols, _ = wl.expert_dims(shape, name)
        W[name] = torch.empty((n, rows, cols), dtype=dt, device="cuda")
        jobs += [(name, e) for e in range(n)]
    keep_set = None if keep is None else set(int(e) for e in keep)
    host = {}

    def one(job):
        name, e = job
        a = wl.gen_expert(shape, name, e, seed)
        if keep_set is not None and (name.startswith("Ws") or e in keep_set):
            host[(name, e)] = a
        t = torch.from_numpy(a)
        W[name][e].copy_(t.view(dt) if shape.dtype == "bf16" else t)

    _, ncpu = host_cpu()
    with ThreadPoolExecutor(max(4, min(32, ncpu))) as ex:
        list(ex.map(one, jobs))
    torch.cuda.synchronize()
    return W, host


def to_dev(torch, a, shape):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if shape.dtype == "bf16":
        t = t.view(torch.bfloat16)
    return t.cuda()


def traffic_for(workload):
    src = os.path.join(ROOT, "mixture_experts_sparse_02_b300", "csrc", "gemm_tc.cu")
    if NCU_TRAFFIC["code_sha256"] and os.path.exists(src) and _code_sha256(src) == NCU_TRAFFIC["code_sha256"]:
        return NCU_TRAFFIC["bytes_per_launch"].get(workload)
    return None


def gemm_variant(shape):
    """Which grouped-GEMM kernel the library runs for the routed W1/W2 + SwiGLU GEMM of this
    workload: the library's rule (the token-wide CTA-pair kernel with wide tiles when expert
    blocks average >= 128 rows, else single CTAs; f32 layers run on CUDA cores; MOE_GEMM_KERNEL
    forces one)."""
    if shape.dtype != "bf16":
        return "simt"
    forced = os.environ.get("MOE_GEMM_KERNEL")
    if forced in ("single", "pair", "tpair", "tpairw"):
        return forced
    return "tpairw" if shape.T * shape.k >= 128 * shape.E else "single"


KERNEL_NAMES = {"pair": "grouped_gemm_pair_kernel<EPI_SWIGLU>",
                "tpair": "grouped_gemm_tpair_kernel<EPI_SWIGLU, false>",
                "tpairw": "grouped_gemm_tpair_kernel<EPI_SWIGLU, true>",
                "single": "grouped_gemm_kernel<EPI_SWIGLU>",
                "simt": "simt_swiglu_f32 (CUDA cores, float32)"}


def measure_workload(args, shape, world, rank, pk, headline):
    """One workload on this rank's GPU: W warm-up steps, K timed steps of moe_forward_profiled
    (L2 flushed before each), the per-stage split, the end-to-end host-buffer runs and the
    CPU-oracle sample.  Returns the record (the headline JSON line's fields)."""
    import torch
    from mixture_experts_sparse_02_b300 import moe

    want_cpu = rank == 0 and world == 1 and not args.no_cpu_baseline
    n_tok = sample_tokens(args, shape)
    # replicated weights (seed 0); each rank draws its own tokens
    x_host = wl.gen_x(shape, 0 if rank == 0 else 1000 + rank)
    Wg_host = wl.gen_router(shape, 0)
    lb_np = wl.gen_logit_bias(shape, 0)
    keep = oracle_experts_needed(shape, x_host[:n_tok], Wg_host, lb_np) if want_cpu else None
    t_gen = time.perf_counter()
    W, W_host = upload_weights(shape, torch, 0, keep)
    gen_s = time.perf_counter() - t_gen
    x = to_dev(torch, x_host, shape)
    W_g = to_dev(torch, Wg_host, shape)
    lb = None if lb_np is None else torch.from_numpy(lb_np).cuda()
    cfg = moe.config_from_shape(shape)
    ws = torch.empty((moe.workspace_bytes(cfg),), dtype=torch.uint8, device="cuda")
    dt = torch.bfloat16 if shape.dtype == "bf16" else torch.float32
    y = torch.empty((shape.T, shape.d), dtype=dt, device="cuda")
    flush = torch.empty((FLUSH_BYTES,), dtype=torch.uint8, device="cuda")
    Ws = dict(Ws1=W.get("Ws1"), Ws2=W.get("Ws2"), Ws3=W.get("Ws3"))

    def step(events=None):
        moe.forward(cfg, x, W_g, W["W1"], W["W2"], W["W3"], y, ws, logit_bias=lb, events=events, **Ws)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    if moe.get_device_error() != 0:
        raise RuntimeError("device error word set during warm-up (%s)" % shape.name)

    # timed: the production call, moe_forward, bracketed by events on the launching stream (no
    # events between its kernels, so each may start while the previous one finishes).  The timed
    # steps start IDLE_BEFORE_TIMED_S after the warm-up steps (the clock sampler's start-up), as
    # the measured bf16 and copy peaks start from an idle GPU; started right after the warm-ups,
    # the power cap lengthens the steps of the long layers (recorded in "timing").
    tev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    launches = 0
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(torch.cuda.current_device()) as clk:
        clk.mark_start()
        for i in range(args.steps):
            flush.zero_()
            tev[i][0].record()
            step()
            tev[i][1].record()
            launches += moe.last_launch_count()
        torch.cuda.synchronize()
        clk.mark_end()
    barrier(world)
    step_ms = [a.elapsed_time(b) for a, b in tev]
    # stage split: moe_forward_profiled, the same kernels with events at the stage boundaries
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(moe.MOE_NUM_STAGES + 1)] for _ in range(args.steps)]
    for i in range(args.steps):
        flush.zero_()
        step(evs[i])
    torch.cuda.synchronize()
    stage_ms = [[evs[i][j].elapsed_time(evs[i][j + 1]) for j in range(moe.MOE_NUM_STAGES)]
                for i in range(args.steps)]
    total_s = sum(step_ms) / 1e3
    total_s_max = max_over_ranks(total_s, world, device="cuda")
    value = shape.T * args.steps * world / total_s_max
    mean_stage = [statistics.mean(s[j] for s in stage_ms) for j in range(moe.MOE_NUM_STAGES)]
    stages = dict(zip(moe.STAGE_NAMES, [round(v, 4) for v in mean_stage]))

    # algorithmic work: W1/W2 + SwiGLU 4 d d_ff per routed row, W3 2 d d_ff, shared 6 d d_ffs per token
    N = shape.T * shape.k
    fl_w12 = 4.0 * N * shape.d * shape.d_ff
    fl_w3 = 2.0 * N * shape.d * shape.d_ff
    fl_sh = 6.0 * shape.T * shape.d * shape.d_ff_shared * shape.n_shared
    t_w12, t_w3, t_sh = mean_stage[2] / 1e3, mean_stage[3] / 1e3, mean_stage[4] / 1e3
    peak = pk["bf16_tflops"]
    ach = fl_w12 / t_w12 / 1e12
    expert_tflops = (fl_w12 + fl_w3 + fl_sh) / (t_w12 + t_w3 + t_sh) / 1e12
    variant = gemm_variant(shape)
    if shape.dtype == "bf16":
        traffic = traffic_for(shape.name)
        roof = {"bound": "tensor", "kernel": KERNEL_NAMES[variant] + " (W1/W2 + SiLU*mul)",
                "achieved": round(ach, 2), "peak": peak, "unit": "TFLOP/s", "frac": round(ach / peak, 4),
                "peak_kind": "bf16 dense burst (%s)" % pk["source"], "traffic": traffic,
                "traffic_unit": "bytes per launch (dram read + write)", "algorithmic_flops_per_launch": fl_w12}
        if traffic:
            # the same launch against the copy bandwidth: the bound at the ridge (DeepSeek-V3 shapes)
            gbs = traffic / t_w12 / 1e9
            roof.update({"dram_gbs": round(gbs, 1), "dram_frac": round(gbs / pk["hbm_gbs"], 4),
                         "dram_peak_gbs": pk["hbm_gbs"]})
        eg = {"tflops": round(expert_tflops, 2), "frac_of_peak": round(expert_tflops / peak, 4), "peak_tflops": peak,
              "w12_ms": round(mean_stage[2], 4), "w3_ms": round(mean_stage[3], 4), "shared_ms": round(mean_stage[4], 4)}
    else:
        roof = {"bound": "latency", "kernel": KERNEL_NAMES[variant], "achieved": round(ach, 4), "peak": None,
                "unit": "TFLOP/s", "frac": None, "traffic": None,
                "note": "float32 correctness workload: a few microseconds per kernel, bound by launch latency"}
        eg = {"tflops": round(expert_tflops, 4), "frac_of_peak": None}

    # decode-shaped batch with the same weights (T = 16 tokens): touched-expert weight bytes / time
    decode = None
    if headline and shape.name == DEFAULT_WORKLOAD and not args.no_decode:
        dshape = wl.WORKLOADS[DECODE_WORKLOAD]
        dcfg = moe.config_from_shape(dshape)
        dws = torch.empty((moe.workspace_bytes(dcfg),), dtype=torch.uint8, device="cuda")
        dx = x[: dshape.T].contiguous()
        dy = torch.empty((dshape.T, dshape.d), dtype=dt, device="cuda")
        counts = torch.empty((dshape.E,), dtype=torch.int32, device="cuda")
        dev_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
        for i in range(args.warmup + args.steps):
            flush.zero_()
            if i >= args.warmup:
                dev_ev[i - args.warmup][0].record()
            moe.forward(dcfg, dx, W_g, W["W1"], W["W2"], W["W3"], dy, dws, logit_bias=lb, counts_out=counts)
            if i >= args.warmup:
                dev_ev[i - args.warmup][1].record()
        torch.cuda.synchronize()
        dms = statistics.mean(a.elapsed_time(b) for a, b in dev_ev)
        touched = int((counts.cpu() > 0).sum())
        wbytes = touched * 3 * dshape.d * dshape.d_ff * 2 + dshape.d * dshape.E * 2
        gbs = wbytes / (dms / 1e3) / 1e9
        decode = {"workload": DECODE_WORKLOAD, "T": dshape.T, "ms_per_step": round(dms, 4),
                  "touched_experts": touched, "touched_weight_bytes": wbytes, "hbm_gbs": round(gbs, 1),
                  "peak_gbs": pk["hbm_gbs"], "frac": round(gbs / pk["hbm_gbs"], 4)}
        del dws, dx, dy

    # end to end through the public calls with host buffers (pinned), copies inside the timed region
    e2e = None
    if not args.no_e2e:
        xh = torch.from_numpy(np.ascontiguousarray(x_host))
        xh = (xh.view(torch.bfloat16) if shape.dtype == "bf16" else xh).pin_memory()
        yh = [torch.empty((shape.T, shape.d), dtype=dt).pin_memory() for _ in range(2)]
        nbytes = shape.T * shape.d * (2 if shape.dtype == "bf16" else 4)
        # (1) moe_forward_host: copy in, layer, copy out, wait; one step after the other
        for _ in range(max(1, args.warmup)):
            moe.forward_host(cfg, xh, W_g, W["W1"], W["W2"], W["W3"], yh[0], ws, logit_bias=lb, **Ws)
        barrier(world)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(args.steps):
            moe.forward_host(cfg, xh, W_g, W["W1"], W["W2"], W["W3"], yh[0], ws, logit_bias=lb, **Ws)
        torch.cuda.synchronize()
        sync_s = max_over_ranks(time.perf_counter() - t0, world, device="cuda")
        # (2) moe_forward_host_async on two streams, each with its own workspace and output
        # buffer: one step's host copies overlap the other step's kernels
        ws2 = torch.empty_like(ws)
        wss = [ws, ws2]
        streams = [torch.cuda.Stream(), torch.cuda.Stream()]
        torch.cuda.synchronize()
        for i in range(max(2, args.warmup)):
            moe.forward_host_async(cfg, xh, W_g, W["W1"], W["W2"], W["W3"], yh[i % 2], wss[i % 2], logit_bias=lb,
                                   stream=streams[i % 2], **Ws)
        for st_ in streams:
            st_.synchronize()
        barrier(world)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for i in range(args.steps):
            moe.forward_host_async(cfg, xh, W_g, W["W1"], W["W2"], W["W3"], yh[i % 2], wss[i % 2], logit_bias=lb,
                                   stream=streams[i % 2], **Ws)
        for st_ in streams:
            st_.synchronize()
        e2e_s = max_over_ranks(time.perf_counter() - t0, world, device="cuda")
        del ws2
        e2e = {"value": shape.T * args.steps * world / e2e_s, "unit": "tokens/s", "h2d_bytes_per_step": nbytes,
               "d2h_bytes_per_step": nbytes,
               "call": "moe_forward_host_async on two alternating streams (one step's copies overlap the "
                       "other step's kernels); all copies inside the timed region",
               "sync": {"value": shape.T * args.steps * world / sync_s, "unit": "tokens/s",
                        "call": "moe_forward_host (copy in, layer, copy out, wait; step after step)"}}

    # CPU oracle baseline on a bounded sample (rank 0 at N = 1 only)
    cpu = None
    if want_cpu:
        get_w = lambda name, e: wl.to_f64(W_host[(name, e)], shape.dtype)
        cpu = cpu_record(shape, oracle_sample(shape, x_host[:n_tok], Wg_host, lb_np, get_w), n_tok)

    err = moe.get_device_error()
    rec = {"value": round(value, 1), "unit": "tokens/s", "ms_per_step": round(1e3 * total_s_max / args.steps, 4),
           "dtype": shape.dtype, "config": workload_config(shape, world), "roofline": roof, "expert_gemm": eg,
           "decode": decode, "stages_ms": stages,
           "stages_from": "moe_forward_profiled (same kernels, events at the stage boundaries)",
           "step_ms": {"min": round(min(step_ms), 4), "median": round(statistics.median(step_ms), 4),
                       "max": round(max(step_ms), 4)},
           "timing": {"warmup_then_idle_s": IDLE_BEFORE_TIMED_S, "l2": "flushed before every step",
                      "clock": "CUDA events on the launching stream"},
           "e2e": e2e, "cpu_baseline": cpu, "gpu_launches": launches,
           "clocks": clk.summary(), "device_error_word": err, "weights_drawn_s": round(gen_s, 1)}
    del W, W_host, x, W_g, lb, ws, y, flush
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return rec


def run_ours(args, shape, world, rank, local):
    import torch
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    pk = peaks()
    head = measure_workload(args, shape, world, rank, pk, headline=True)
    extras = {}
    if world == 1 and not args.override:
        for name in [w for w in args.workloads.split(",") if w and w != "none"]:
            if name != shape.name:
                extras[name] = measure_workload(args, wl.WORKLOADS[name], world, rank, pk, headline=False)
    if rank == 0:
        line = {"metric": METRIC, "value": head["value"], "unit": "tokens/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["ms_per_step"],
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": head["dtype"],
                "data": "synthetic (seeded: x ~ N(0,1), weights ~ N(0,1/fan_in); per-rank tokens, replicated weights)"}
        line.update({k: v for k, v in head.items() if k not in ("value", "unit", "ms_per_step", "dtype")})
        line["workloads"] = extras
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(wl.WORKLOADS))
    ap.add_argument("--workloads", default=",".join(EXTRA_WORKLOADS),
                    help="further workloads measured after the headline one at N = 1 (comma list, or 'none')")
    ap.add_argument("--ref-tokens", type=int, default=0, help="tokens per CPU-oracle sample (0: per workload)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--override", default="", help="size overrides for profiling runs, e.g. T=2048,E=2,k=1")
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.impl == "ours":
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    world, rank, local = dist_env()
    shape = wl.WORKLOADS[args.workload]
    if args.override:
        kv = dict(item.split("=") for item in args.override.split(","))
        shape = shape.replace(name=shape.name + "[" + args.override + "]", **{k: int(v) for k, v in kv.items()})
    if args.impl == "reference":
        return run_reference(args, shape, world, rank)
    return run_ours(args, shape, world, rank, local)


if __name__ == "__main__":
    sys.exit(main())
