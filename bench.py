"""Benchmark of the MoE FFN layer forward (DeepSeek-V3 shape) on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--config v3|decode|skewed|tiny|v3_e32|sweep|sweep_mx] [--mx]
                    [--backward] [--tiling auto|single|pair|swap]

One step is one pass of the whole hot path over one batch: router logits, routing,
permutation, 1x128 quantisation, row gather, gate/up grouped GEMM with fused SwiGLU and
requantisation, down grouped GEMM and combine.  In the skewed-load configuration a step
is the whole procedure of that workload: starting from its Zipf bias, a forward pass,
the aux-loss-free bias update, and a second forward pass with the updated bias (2T
tokens per step).  Rank 0 prints one JSON line.  Under torchrun each rank runs its own replica on its own GPU and
its own tokens (weak scaling, no collective on the data path); the time is the max over
ranks.

--impl reference times the CPU oracle (numpy, float64) on a bounded sample of the same
workload: each step routes one token and runs its experts, one token at a time.

Inputs are synthetic and seeded (workloads.py).  The weights of the experts a step
touches (several GB of E4M3) are larger than L2 and are streamed from HBM every step,
so no L2 flush is needed between steps.
"""

import argparse
import hashlib
import json
import os
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np
import torch

import workloads

METRIC = "MoE-layer fwd tokens/s & FP8 TFLOPS at V3 shape; % of B300 FP8/HBM roofline"
GAMMA = 0.001
# the kernel sources the committed DRAM-traffic figure was measured with
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "fp8_gemm_gate_up_v3_traffic.txt")
GEMM_SOURCES = ["fp8_block_scaled_bias_b300/csrc/gemm_fp8.cu",
                "fp8_block_scaled_bias_b300/csrc/common.cuh"]


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", choices=["v3", "decode", "skewed", "tiny", "v3_e32", "decode_e32",
                                         "sweep", "sweep_mx"],
                    default="v3")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--mx", action="store_true",
                    help="layer configs: the MX-native variant (power-of-two scales applied by "
                         "the tensor core) instead of FP32 scales with software promotion")
    ap.add_argument("--backward", action="store_true",
                    help="layer configs: time a training step (forward + expert backward)")
    ap.add_argument("--tiling", choices=["auto", "single", "pair", "swap"], default="auto",
                    help="CTA tiling of the FP32-scale grouped GEMM (moe_set_gemm_tiling)")
    ap.add_argument("--shape", default=None,
                    help="sweep configs only: one M,N,K instead of the five sweep shapes")
    return ap.parse_args()


# ---- distributed plumbing ----------------------------------------------------------------

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    return rank, world, torch.device("cuda", torch.cuda.current_device())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v, world):
    """The largest of the ranks' values (the slowest rank's time): one all-reduce on the
    host-side timing result, not on the data path."""
    if world == 1:
        return v
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_value(tokens_per_rank, steps, world, ms_max):
    """Whole-job throughput: the tokens every rank processed over the slowest rank's time."""
    return tokens_per_rank * world * steps / (ms_max / 1e3)


# ---- peaks, clocks -----------------------------------------------------------------------

def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        m = json.load(open(p))
        return {"hbm_gbs": float(m["hbm_gbs"]), "bf16_tflops": float(m["bf16_tflops"]),
                "bf16_tflops_sustained": float(m.get("bf16_tflops_sustained", m["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0,
                "source": "fallback"}


class ClockSampler:
    """Samples SM clock and clock-event reasons through NVML while the timed region runs."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
               0x2: "applications_clocks_setting", 0x100: "display_clock_setting"}

    SMI_FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.sw_power_cap,"
                  "clocks_event_reasons.hw_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
                  "clocks_event_reasons.hw_thermal_slowdown")

    def __init__(self, index, period=0.01):
        self.samples, self.reasons, self.period, self.index = [], set(), period, index
        self._stop = threading.Event()
        self.proc = None
        try:
            import pynvml
            pynvml.nvmlInit()
            self.nv = pynvml
            self.h = pynvml.nvmlDeviceGetHandleByIndex(index)
            self.max_mhz = pynvml.nvmlDeviceGetMaxClockInfo(self.h, pynvml.NVML_CLOCK_SM)
        except Exception:
            self.nv = None
            self.max_mhz = None

    def _run(self):
        nv = self.nv
        while not self._stop.is_set():
            try:
                self.samples.append(nv.nvmlDeviceGetClockInfo(self.h, nv.NVML_CLOCK_SM))
                r = nv.nvmlDeviceGetCurrentClocksEventReasons(self.h)
                for bit, name in self.REASONS.items():
                    if r & bit:
                        self.reasons.add(name)
            except Exception:
                pass
            time.sleep(self.period)

    def __enter__(self):
        if self.nv is not None:
            self._t = threading.Thread(target=self._run, daemon=True)
            self._t.start()
        else:                      # no NVML binding: sample with nvidia-smi instead
            import subprocess
            try:
                self.proc = subprocess.Popen(
                    ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.SMI_FIELDS,
                     "--format=csv,noheader,nounits", "-lms", "20"],
                    stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
                # wait for the sampler's first line (taken before the timed region, not
                # kept) so that even a short timed region is sampled
                self.proc.stdout.readline()
            except Exception:
                self.proc = None
        return self

    def __exit__(self, *a):
        if self.nv is not None:
            self._stop.set()
            self._t.join()
        elif self.proc is not None:
            self.proc.terminate()
            out, _ = self.proc.communicate(timeout=10)
            names = ("sw_power_cap", "hw_slowdown", "sw_thermal_slowdown", "hw_thermal_slowdown")
            for line in out.splitlines():
                f = [v.strip() for v in line.split(",")]
                if len(f) < 6:
                    continue
                try:
                    self.samples.append(float(f[0]))
                    self.max_mhz = float(f[1])
                except ValueError:
                    continue
                for name, v in zip(names, f[2:6]):
                    if v.lower() == "active":
                        self.reasons.add(name)

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": sorted(self.reasons),
                    "samples": 0}
        return {"sm_mhz": statistics.median(self.samples), "sm_max_mhz": self.max_mhz,
                "reasons": sorted(self.reasons), "samples": len(self.samples)}


def gemm_source_hash():
    h = hashlib.sha256()
    for p in GEMM_SOURCES:
        h.update(open(os.path.join(ROOT, p), "rb").read())
    return h.hexdigest()[:16]


def committed_traffic():
    """DRAM bytes per gate/up launch from the committed ncu summary, if it was taken with
    the current kernel source; else None."""
    try:
        t = {}
        for line in open(TRAFFIC_FILE):
            if ":" in line and not line.startswith("#"):
                k, v = line.split(":", 1)
                t[k.strip()] = v.strip()
    except OSError:
        return None
    if t.get("kernel_source_sha256_16") != gemm_source_hash():
        return None
    v = t.get("dram_bytes_per_launch_v3")
    return int(v) if v else None


# ---- our arm -----------------------------------------------------------------------------

def gate_up_bytes(cfg, counts_np, T):
    """Algorithmic HBM bytes of one gate/up launch: the weights and scales of every expert
    segment with at least one row, the gathered FP8 rows and their scales read once, and
    the FP8 h rows and scales written once."""
    E, d, f = cfg.E, cfg.d, cfg.f
    active = int((counts_np > 0).sum()) + 1                    # + the shared expert
    rows = T * cfg.K + T
    w = active * (2 * f * d + (2 * f // 128) * (d // 128) * 4)
    a = rows * d + rows * (d // 128) * 4
    h = rows * f + rows * (f // 128) * 4
    return w + a + h


def down_bytes(cfg, counts_np, T):
    E, d, f = cfg.E, cfg.d, cfg.f
    active = int((counts_np > 0).sum()) + 1
    rows = T * cfg.K + T
    return active * (d * f + (d // 128) * (f // 128) * 4) + rows * f + rows * (f // 128) * 4 + \
        rows * d * 2


def run_layer(args, cfg, rank, world, dev):
    from fp8_block_scaled_bias_b300 import MoELayer, make_weights
    from fp8_block_scaled_bias_b300.layer import MoELayer as _L

    T = cfg.T
    w = make_weights(cfg, dev, pow2=args.mx)
    x_host = workloads.gen_x(cfg, base_seed=rank).pin_memory()
    x = x_host.to(dev)
    layer = MoELayer(cfg, w, mx=args.mx)
    skewed = cfg.zipf_s > 0
    bias0 = w.bias.clone()
    stages = list(_L.STAGE_LAUNCHES) + (["bias_update"] if skewed else [])
    launches_per_step = (2 * sum(_L.STAGE_LAUNCHES.values()) + 1 if skewed
                         else sum(_L.STAGE_LAUNCHES.values()))

    def procedure(mk=None):
        if skewed:
            w.bias.copy_(bias0)             # every step starts from the workload's own bias
            layer.forward(x, mark=mk)
            layer.bias_update(GAMMA)
            if mk:
                mk("bias_update")
        layer.forward(x, mark=mk)

    def step(marks=None):
        mk = None
        if marks is not None:
            def mk(name):
                e = torch.cuda.Event(enable_timing=True)
                e.record()
                marks.append((name, e))
        procedure(mk)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    layer.check_status()

    # device-resident timed region
    all_marks = []
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(dev.index) as clocks:
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record()
        for _ in range(args.steps):
            marks = [("start", None)]
            ev = torch.cuda.Event(enable_timing=True)
            ev.record()
            marks[0] = ("start", ev)
            step(marks)
            all_marks.append(marks)
        t1.record()
        torch.cuda.synchronize()
    barrier(world)
    ms_total = max_over_ranks(t0.elapsed_time(t1), world)
    layer.check_status()
    stage_ms = {s: 0.0 for s in stages}
    for marks in all_marks:
        for (n0, e0), (n1, e1) in zip(marks[:-1], marks[1:]):
            stage_ms[n1] += e0.elapsed_time(e1)
    stage_ms = {k: v / args.steps for k, v in stage_ms.items()}

    # End to end through the public API: every step copies its input x from pinned host
    # memory and reads its output y back to pinned host memory.  x and y are double
    # buffered so that step i+1's input copy and step i-1's output copy run on their own
    # streams while step i computes; events order each copy against the compute that
    # uses or overwrites its buffer.
    y_host = [torch.empty(T, cfg.d, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    xb = [torch.empty_like(x) for _ in range(2)]
    yb = [torch.empty(T, cfg.d, dtype=torch.bfloat16, device=dev) for _ in range(2)]
    comp = torch.cuda.current_stream()
    h2d, d2h = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()
    x_ready, x_free = [ev(), ev()], [ev(), ev()]
    y_ready, y_free = [ev(), ev()], [ev(), ev()]

    def e2e_step(i):
        j = i % 2
        with torch.cuda.stream(h2d):
            if i >= 2:
                h2d.wait_event(x_free[j])              # step i-2 has read this buffer
            xb[j].copy_(x_host, non_blocking=True)
            x_ready[j].record(h2d)
        comp.wait_event(x_ready[j])
        if i >= 2:
            comp.wait_event(y_free[j])                 # step i-2's output has left
        if skewed:
            w.bias.copy_(bias0)
            layer.forward(xb[j])
            layer.bias_update(GAMMA)
        layer.forward(xb[j], out=yb[j])
        x_free[j].record(comp)
        y_ready[j].record(comp)
        with torch.cuda.stream(d2h):
            d2h.wait_event(y_ready[j])
            y_host[j].copy_(yb[j], non_blocking=True)
            y_free[j].record(d2h)

    for i in range(2):                                 # warm the streams and events
        e2e_step(i)
    torch.cuda.synchronize()
    barrier(world)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(h2d)
    for i in range(args.steps):
        e2e_step(i)
    comp.wait_stream(d2h)
    e1.record(comp)
    torch.cuda.synchronize()
    barrier(world)
    ms_e2e = max_over_ranks(e0.elapsed_time(e1), world)
    layer.check_status()
    assert torch.equal(y_host[(args.steps - 1) % 2], yb[(args.steps - 1) % 2].cpu())

    counts = layer.counts.cpu().numpy()
    return dict(ms_total=ms_total, stage_ms=stage_ms, ms_e2e=ms_e2e, clocks=clocks.summary(),
                counts=counts, launches=launches_per_step * args.steps,
                forwards_per_step=2 if skewed else 1,
                h2d=x_host.numel() * 2, d2h=y_host[0].numel() * 2, layer=layer, weights=w,
                x=x_host)


def _oracle_token_times(payload):
    """Worker (spawned with one BLAS/OpenMP thread): time oracle.moe_layer_tokens on one
    token per step."""
    import oracle
    cfg, tokens, xr, cen, bias, q, steps, pow2 = payload
    times = []
    for s in range(steps):
        i = s % len(tokens)
        t0 = time.perf_counter()
        oracle.moe_layer_tokens([tokens[i]], xr[i:i + 1], cen, bias, None, cfg.n_groups,
                                cfg.topk_groups, cfg.K, expert_quantised=q.__getitem__,
                                pow2=pow2)
        times.append(time.perf_counter() - t0)
    return times


class _WorkerThreads:
    """Within this block, newly started processes run numpy with `n` threads (the
    variables are read when a process imports numpy; this process is not affected)."""
    KEYS = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")

    def __init__(self, n):
        self.n = n

    def __enter__(self):
        self.old = {k: os.environ.get(k) for k in self.KEYS}
        for k in self.KEYS:
            os.environ[k] = str(self.n)

    def __exit__(self, *a):
        for k, v in self.old.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v


def _spawn_pool(workers):
    import concurrent.futures as cf
    import multiprocessing as mp
    return cf.ProcessPoolExecutor(max_workers=workers, mp_context=mp.get_context("spawn"))


def cpu_baseline(cfg, cen, bias, x_host, n_tokens=4, steps=None, pow2=False):
    """The oracle, as it stands, on a bounded sample: n_tokens tokens of the workload, one
    at a time through oracle.moe_layer_tokens (routing in float64/float32, every expert
    block-scaled GEMM exact in float64), in one process with one thread.  Expert weights
    are generated from the same seeds and quantised by the oracle in spawned worker
    processes before timing starts."""
    import oracle

    rng = np.random.default_rng(7)
    tokens = sorted(rng.choice(cfg.T, n_tokens, replace=False).tolist())
    xr = x_host.float().numpy()[tokens]
    z = oracle.router_logits(xr, cen)
    idx, _ = oracle.route(z, bias, cfg.n_groups, cfg.topk_groups, cfg.group_topn, cfg.K)
    need = sorted(set(int(e) for r in idx for e in r) | {cfg.E})
    mats = []
    for e in need:
        mats.extend(t.cpu().numpy() for t in workloads.gen_expert_f32(cfg, e, device="cuda"))
    workers = max(1, min(16, (os.cpu_count() or 2) - 1))
    with _WorkerThreads(1):
        with _spawn_pool(workers) as pool:
            quant = list(pool.map(oracle.quant_128x128_pow2 if pow2 else oracle.quant_128x128,
                                  mats))
        q = {e: tuple(a for j in range(3) for a in quant[3 * i + j]) for i, e in enumerate(need)}
        del mats, quant
        steps = steps or n_tokens
        with _spawn_pool(1) as pool:
            times = pool.submit(_oracle_token_times,
                                (cfg, tokens, xr, cen, bias, q, steps, pow2)).result()
    return dict(value=len(times) / sum(times), times=times, tokens=tokens, cores=1)


def gate_up_flops(cfg, T):
    """Algorithmic FP8 FLOPs of one gate/up launch (no padding): every routed and shared
    row times the [2f, d] gate/up weights."""
    return 2 * (T * cfg.K + T) * (2 * cfg.f) * cfg.d


def fp8_peak_for(pk, clocks):
    """FP8 dense peak for a kernel timed in a region with these sampled clocks: 2 x the
    measured BF16 peak (the nominal FP8/BF16 ratio), burst unless the samples show the
    power cap or a median SM clock under 95% of the maximum, where the sustained figure
    applies.  Returns (TFLOP/s, note)."""
    capped = "sw_power_cap" in (clocks.get("reasons") or [])
    mhz, mx = clocks.get("sm_mhz"), clocks.get("sm_max_mhz")
    slow = bool(mhz and mx and mhz < 0.95 * mx)
    if capped or slow:
        return 2.0 * pk["bf16_tflops_sustained"], "2 x measured sustained bf16 (clocks: power cap)"
    return 2.0 * pk["bf16_tflops"], "2 x measured burst bf16 (clocks at max, no power cap)"


def kernel_roofline(name, bytes_, flops, ms, pk, fp8_peak):
    """Roofline of one kernel: the bound is whichever of HBM bytes / measured HBM
    bandwidth and FLOPs / FP8 peak takes longer; achieved and peak are in that unit."""
    t_hbm = bytes_ / (pk["hbm_gbs"] * 1e9)
    t_tc = flops / (fp8_peak * 1e12)
    if t_hbm >= t_tc:
        ach = bytes_ / (ms / 1e3) / 1e9
        r = {"kernel": name, "bound": "hbm", "achieved": round(ach, 1), "peak": pk["hbm_gbs"],
             "unit": "GB/s", "frac": round(ach / pk["hbm_gbs"], 4)}
    else:
        ach = flops / (ms / 1e3) / 1e12
        r = {"kernel": name, "bound": "tensor", "achieved": round(ach, 1), "peak": fp8_peak,
             "unit": "TFLOP/s", "frac": round(ach / fp8_peak, 4)}
    r.update({"algorithmic_bytes": bytes_, "algorithmic_flops": flops,
              "hbm_frac": round(bytes_ / (ms / 1e3) / 1e9 / pk["hbm_gbs"], 4),
              "tensor_frac": round(flops / (ms / 1e3) / 1e12 / fp8_peak, 4),
              "roofline_ms": round(1e3 * max(t_hbm, t_tc), 4), "measured_ms": round(ms, 4)})
    return r


def main_ours(args, cfg, rank, world, dev):
    pk = peaks()
    r = run_layer(args, cfg, rank, world, dev)
    T, K = cfg.T, args.steps
    fw = r["forwards_per_step"]
    ms_step = r["ms_total"] / K
    tokens_s = weak_scaling_value(fw * T, K, world, r["ms_total"])
    flops = cfg.flops()
    st = r["stage_ms"]
    gu_bytes = gate_up_bytes(cfg, r["counts"], T)
    gu_ms = st["gate_up"] / fw
    fp8_peak, peak_note = fp8_peak_for(pk, r["clocks"])
    gemm_ms = (st["gate_up"] + st["down"]) / fw
    roof = kernel_roofline(gate_up_kernel_name(cfg, T, args.mx, _lib_tiling()), gu_bytes,
                           gate_up_flops(cfg, T), gu_ms, pk, fp8_peak)
    roof["traffic"] = committed_traffic() if cfg.name == "v3" and not args.mx else None
    roof["peak_source"] = pk["source"] + (f" ({peak_note})" if roof["bound"] == "tensor"
                                          else " (copy)")
    roof["fp8_peak_tflops"] = fp8_peak
    layer_bytes = gu_bytes + down_bytes(cfg, r["counts"], T)
    workload = (f"DeepSeek-V3-shape MoE layer fwd ({cfg.name}): T={T}, d_model={cfg.d}, "
                f"{cfg.E} routed experts in {cfg.n_groups} groups, top-{cfg.K} of at most "
                f"{cfg.topk_groups} groups, d_ffn={cfg.f}, 1 shared expert")
    if fw == 2:
        workload += (f"; Zipf({cfg.zipf_s}) bias; each step: forward, bias update "
                     f"gamma={GAMMA}, forward (2T tokens)")
    if args.mx:
        workload += ("; MX-native variant: power-of-two block scales applied by the tensor "
                     "core (tcgen05 kind::mxf8f6f4)")
    out = {
        "metric": METRIC, "value": round(tokens_s, 1), "unit": "tokens/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "fp8_e4m3", "data": "synthetic",
        "config": {"workload": workload,
                   "tokens_per_gpu": T, "parallelism": f"replicas x{world}",
                   "l2": "inputs larger than L2 (all touched expert weights streamed from HBM "
                         "each step)"},
        "fp8_tflops": round(fw * flops * world * K / (r["ms_total"] / 1e3) / 1e12, 1),
        "gemm_fp8_tflops": round(flops / (gemm_ms / 1e3) / 1e12, 1),
        "roofline": roof,
        "layer_roofline": {
            "hbm_bytes": layer_bytes,
            "hbm_frac": round(fw * layer_bytes / (ms_step / 1e3) / 1e9 / pk["hbm_gbs"], 4),
            "tensor_frac": round(fw * flops / (ms_step / 1e3) / 1e12 / fp8_peak, 4),
            "roofline_ms": round(1e3 * fw * max(layer_bytes / (pk["hbm_gbs"] * 1e9),
                                                flops / (fp8_peak * 1e12)), 4),
            "fp8_peak_tflops": fp8_peak, "fp8_peak_note": peak_note},
        "active_experts": int((r["counts"] > 0).sum()),
        "stage_ms": {k: round(v, 4) for k, v in st.items()},
        "e2e": {"value": round(fw * T * world * K / (r["ms_e2e"] / 1e3), 1), "unit": "tokens/s",
                "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"]},
        "gpu_launches": r["launches"],
        "gemm_tiling": _lib_tiling(),
        "clocks": r["clocks"],
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cb = cpu_baseline(cfg, r["weights"].centroids.cpu().numpy(),
                          r["weights"].bias.cpu().numpy(), r["x"], pow2=args.mx)
        out["cpu_baseline"] = {"value": round(cb["value"], 4), "unit": "tokens/s", "cores": cb["cores"],
                               "kind": "oracle",
                               "sample": f"{len(cb['times'])} tokens of this workload, one at a time "
                                         f"through the numpy oracle (tokens {cb['tokens']}); expert "
                                         f"weights pre-quantised outside the timing"}
    if rank == 0:
        print(json.dumps(out), flush=True)


def main_backward(args, cfg, rank, world, dev):
    """A training step of the layer's experts: the training forward (SwiGLU inputs cached
    in FP8) and the expert backward (Dgrad and Wgrad of all three matrices, 128x1
    regrouping, SwiGLU recompute) from a seeded dy.  One JSON line; stage times from CUDA
    events; the roofline is the gate/up Wgrad's."""
    from fp8_block_scaled_bias_b300 import MoELayer, make_weights
    pk = peaks()
    T = cfg.T
    w = make_weights(cfg, dev)
    x = workloads.gen_x(cfg, base_seed=rank).to(dev)
    g = torch.Generator().manual_seed(1000 + rank)
    dy = (torch.randn(T, cfg.d, generator=g) * 0.1).to(torch.bfloat16).to(dev)
    layer = MoELayer(cfg, w, train=True)
    layer.transposed_weights()                              # setup, not timed

    def step(marks=None):
        mk = None
        if marks is not None:
            def mk(name):
                e = torch.cuda.Event(enable_timing=True)
                e.record()
                marks.append((name, e))
        layer.forward(x, mark=mk)
        return layer.backward(dy, mark=mk)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    layer.check_status()
    all_marks = []
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(dev.index) as clocks:
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record()
        for _ in range(args.steps):
            e = torch.cuda.Event(enable_timing=True)
            e.record()
            marks = [("start", e)]
            out = step(marks)
            all_marks.append(marks)
        t1.record()
        torch.cuda.synchronize()
    barrier(world)
    ms_total = max_over_ranks(t0.elapsed_time(t1), world)
    layer.check_status()
    stage_ms = {}
    for marks in all_marks:
        for (n0, e0), (n1, e1) in zip(marks[:-1], marks[1:]):
            stage_ms[n1] = stage_ms.get(n1, 0.0) + e0.elapsed_time(e1) / args.steps
    counts = layer.counts.cpu().numpy()
    rows, kpad = layer.rows, int(out["pad"][-1].item())
    d, f, G = cfg.d, cfg.f, cfg.E + 1
    cl = clocks.summary()
    fp8_peak, peak_note = fp8_peak_for(pk, cl)
    wg_flops = 2 * rows * 2 * f * d
    wg_bytes = 2 * f * kpad + d * kpad + kpad // 128 * (2 * f + d) * 4 + G * 2 * f * d * 4
    roof = kernel_roofline("fp8_mx_gemm_kernel<F32> (gate/up Wgrad)", wg_bytes, wg_flops,
                           stage_ms["gate_up_wgrad"], pk, fp8_peak)
    roof["traffic"] = None
    train_flops = 3 * cfg.flops()               # forward + Dgrad + Wgrad of each matrix
    ms_step = ms_total / args.steps
    out_line = {
        "metric": "MoE-layer training step (forward + expert backward) tokens/s",
        "value": round(T * world * args.steps / (ms_total / 1e3), 1), "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms_step, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "fp8_e4m3", "data": "synthetic",
        "config": {"workload": f"DeepSeek-V3-shape MoE layer ({cfg.name}): T={T}, d_model={d}, "
                               f"{cfg.E} routed experts, top-{cfg.K}, d_ffn={f}, 1 shared "
                               f"expert; training forward + expert backward (router and gate "
                               f"gradients not computed); dy ~ N(0, 0.1) BF16",
                   "tokens_per_gpu": T, "parallelism": f"replicas x{world}",
                   "l2": "inputs larger than L2"},
        "fp8_tflops": round(train_flops * world * args.steps / (ms_total / 1e3) / 1e12, 1),
        "roofline": roof,
        "stage_ms": {k: round(v, 4) for k, v in stage_ms.items()},
        "active_experts": int((counts > 0).sum()),
        "gpu_launches": (sum(layer.STAGE_LAUNCHES.values()) + layer.BACKWARD_LAUNCHES) * args.steps,
        "clocks": cl,
    }
    if rank == 0:
        print(json.dumps(out_line), flush=True)


def main_reference(args, cfg, rank, world, dev):
    if rank != 0:
        return
    # the oracle needs only the router and the experts of the sampled tokens, all from
    # the same seeded generators as our arm
    cen = workloads.gen_centroids(cfg).numpy()
    bias = workloads.gen_bias(cfg).numpy()
    x_host = workloads.gen_x(cfg)
    cb = cpu_baseline(cfg, cen, bias, x_host, n_tokens=4, steps=args.warmup + args.steps)
    times = cb["times"][args.warmup:] or cb["times"]
    value = len(times) / sum(times)
    out = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "tokens/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * sum(times) / len(times), 2), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"DeepSeek-V3-shape MoE layer fwd ({cfg.name}): T={cfg.T}, "
                               f"d_model={cfg.d}, {cfg.E} routed experts in {cfg.n_groups} "
                               f"groups, top-{cfg.K}, d_ffn={cfg.f}, 1 shared expert",
                   "tokens_per_gpu": cfg.T, "parallelism": "none (host CPU)"},
        "cpu_baseline": {"value": round(value, 4), "unit": "tokens/s", "cores": cb["cores"],
                         "kind": "oracle",
                         "sample": "each step: one token of the workload through the numpy "
                                   f"oracle (cycling tokens {cb['tokens']})"},
        "e2e": {"value": round(value, 4), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out), flush=True)


def gate_up_kernel_name(cfg, T, mx, tiling):
    """The kernel that runs the gate/up GEMM: segments averaging at most 16 rows (decode
    batches) go to the swapped-operand kernel, in either scale recipe."""
    rows, G = T * cfg.K + T, cfg.E + 1
    if tiling == "swap" or (tiling == "auto" and rows <= 16 * G):
        return "fp8_gemm_swap_kernel<SwiGLU> (gate/up grouped GEMM, weight rows on the MMA M side)"
    if mx:
        return "fp8_mx_gemm_kernel<SwiGLU> (gate/up grouped GEMM)"
    return "fp8_gemm_kernel<SwiGLU> (gate/up grouped GEMM)"


def _lib_tiling():
    from fp8_block_scaled_bias_b300 import load
    return {0: "auto", 1: "single", 2: "pair", 3: "swap"}[load().moe_get_gemm_tiling()]


def main_sweep(args, rank, dev, mx=False):
    """Standalone FP8 block-scaled GEMM sweep (one JSON line per shape); L2 is flushed
    between timed launches.  mx: the MX-native variant (power-of-two scales applied by
    the tensor core) on the same inputs quantised with power-of-two scales."""
    from fp8_block_scaled_bias_b300 import ops
    pk = peaks()
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    shapes = workloads.GEMM_SWEEP
    if args.shape:
        shapes = [tuple(int(v) for v in args.shape.split(","))]
    for (M, N, K) in shapes:
        a = workloads.gen_normal(M, K, sub_seed=31, device="cuda").to(torch.bfloat16)
        b = workloads.gen_normal(N, K, sub_seed=32, device="cuda")
        qa, sa = ops.quant_1x128(a, pow2=mx)
        qb, sb = ops.quant_128x128(b, pow2=mx)
        del a, b
        seg = torch.tensor([0, M], dtype=torch.int32, device=dev)
        C = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
        if mx:
            run = lambda: ops.mx_grouped_gemm(qa, sa, qb[None], sb[None], seg, M, out=C)
        else:
            run = lambda: ops.grouped_gemm(qa, sa, qb[None], sb[None], seg, M, out=C)
        for _ in range(args.warmup):
            flush.zero_()
            run()
        # enough timed launches for the region to last >= 0.5 s (clock samples), at
        # least --steps of them
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(3):
            flush.zero_()
            run()
        e1.record()
        torch.cuda.synchronize()
        per = e0.elapsed_time(e1) / 3
        reps = max(args.steps, int(500.0 / max(per, 1e-3)) + 1)
        ts = []
        with ClockSampler(dev.index) as clocks:
            for _ in range(reps):
                flush.zero_()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                run()
                e1.record()
                ts.append((e0, e1))
            torch.cuda.synchronize()
        ms = statistics.median(e0.elapsed_time(e1) for e0, e1 in ts)
        tf = 2.0 * M * N * K / (ms / 1e3) / 1e12
        cl = clocks.summary()
        fp8_peak, peak_note = fp8_peak_for(pk, cl)
        name = "FP8 MX-scaled GEMM TFLOPS" if mx else "FP8 block-scaled GEMM TFLOPS"
        print(json.dumps({"metric": name, "value": round(tf, 1),
                          "unit": "TFLOP/s", "config": {"workload": f"GEMM sweep M={M} N={N} K={K}",
                                                        "l2": "flushed between launches"},
                          "ms": round(ms, 4), "steps": reps,
                          "roofline": {"bound": "tensor", "achieved": round(tf, 1),
                                       "peak": fp8_peak, "unit": "TFLOP/s",
                                       "frac": round(tf / fp8_peak, 4),
                                       "peak_note": peak_note},
                          "tiling": _lib_tiling(),
                          "clocks": cl}), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        rank = int(os.environ.get("RANK", "0"))
        if rank != 0:
            return
        cfg = workloads.CONFIGS["v3" if args.config in ("sweep", "sweep_mx") else args.config]
        torch.cuda.set_device(0)
        main_reference(args, cfg, 0, 1, torch.device("cuda", 0))
        return
    rank, world, dev = dist_setup()
    import fp8_block_scaled_bias_b300 as pkg
    if not os.path.exists(pkg.LIB_PATH):
        from fp8_block_scaled_bias_b300.build import build
        build()
    lib = pkg.load()
    lib.moe_set_gemm_tiling({"auto": 0, "single": 1, "pair": 2, "swap": 3}[args.tiling])
    if args.config in ("sweep", "sweep_mx"):
        main_sweep(args, rank, dev, mx=args.config == "sweep_mx")
    elif args.backward:
        main_backward(args, workloads.CONFIGS[args.config], rank, world, dev)
    else:
        main_ours(args, workloads.CONFIGS[args.config], rank, world, dev)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
