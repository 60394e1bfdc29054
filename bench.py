"""Benchmark: paged GQA decode step (RoPE + KV append, then decode attention)
on Llama-3.2-1B attention shapes, one JSON line on stdout.

Default workload: batch 32 x 16 layers x 2048-token contexts, 65536 shuffled
16-token pages (2 GiB bf16 pool).  One step = for every layer: append one new token
per sequence (K rotated at its absolute position and written into its page, q
rotated) and decode attention over the sequence's pages -- by default as one
fused kernel (paged_gqa_decode_append); --unfused runs kv_append_rope followed
by paged_gqa_decode.  The pool (2 GiB per step) is larger than L2, so no flush is
needed between steps.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]
                    [--workload batch32|stress256]

Under torchrun (N > 1) every rank runs the same workload on its own GPU
(replicas, weak scaling, no collective on the data path); rank 0 prints the
line with the max elapsed time over ranks.
"""
from __future__ import annotations

import argparse
import datetime as _dt
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)
for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")   # the CPU oracle baseline runs on one core

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads as W  # noqa: E402

METRIC = "paged GQA decode: KV-read GB/s (% of HBM peak), decode tokens/s, µs/layer"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0   # one earlier burst measurement on a GB300


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--workload", choices=["batch32", "stress256", "int8", "int8_stress256",
                                           "mixed8", "single37", "continuous", "prefill",
                                           "argmax"],
                    default="batch32",
                    help="batch32 / stress256: the decode step; int8 / int8_stress256: the same "
                         "step on INT8 K/V pages; mixed8 / single37: one decode launch on the "
                         "batch of 8 mixed lengths (L2 flushed before each launch, warm beside it) "
                         "or the one 37-token sequence (latency); continuous: the 64-request "
                         "continuous-batching mix run to completion; prefill: causal prefill of 8 "
                         "prompts x 1920 tokens; argmax: next-token argmax of 32 x 128256 logits")
    ap.add_argument("--compute", choices=["tensor", "fma"], default="tensor")
    ap.add_argument("--layers", type=int, default=0,
                    help="layers of the workload (0 = its own: 16); fewer layers shrink the pool "
                         "for a profiler capture of the same kernel shape")
    ap.add_argument("--schedule", choices=["auto", "static", "dynamic"], default="auto",
                    help="decode schedule (opts.schedule 2, 0 or 1; auto: dynamic when every SM "
                         "gets at least 512 units of work)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-sustained", action="store_true",
                    help="skip the 2 s sustained window of the headline (profiler runs)")
    ap.add_argument("--unfused", action="store_true",
                    help="run append and decode as two kernels per layer")
    return ap.parse_args()


def effective_schedule(schedule, case, dev):
    """The schedule a decode launch of `case` runs with (include/pkv.h: the
    automatic one is dynamic from PKV_DYNAMIC_MIN_UNITS = 512 units per SM)."""
    if schedule != "auto":
        return schedule
    units = 8 * case.num_seqs * ((int(case.max_seq_len) + 15) // 16)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    return "dynamic" if units >= 512 * sms else "static"


def make_case(name, layers=0):
    case = W.case_batch32() if name in ("batch32", "int8") else W.case_stress()
    if layers and layers != case.num_layers:  # same batch, context and seed, fewer layers
        case = W.case_uniform(case.seed, case.num_seqs, layers, int(case.seq_lens[0]),
                              outlier_frac=case.outlier_frac,
                              name=case.name.replace(f"_l{case.num_layers}_", f"_l{layers}_"))
    return case


# ------------------------------------------------------------- distributed --

def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ clocks --

class ClockSampler:
    """nvidia-smi samples every 200 ms; summarised over a wall-clock window."""
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.proc = None
        self.path = os.path.join("/tmp", f"pkv_clocks_{os.getpid()}.csv")
        try:
            uuid = None
            try:
                uuid = str(torch.cuda.get_device_properties(device_index).uuid)
                if uuid and not uuid.startswith("GPU-"):
                    uuid = "GPU-" + uuid
            except Exception:
                uuid = None
            cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                   "-lms", "200"]
            if uuid:
                cmd += ["-i", uuid]
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(cmd, stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self, t0, t1):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                ts = _dt.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((ts, float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        inside = [r for r in rows if t0 - 0.25 <= r[0] <= t1 + 0.25] or rows
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i, v in enumerate(r[3]) if v == "Active"})
        return {"sm_mhz": statistics.median(r[1] for r in inside),
                "sm_max_mhz": max(r[2] for r in inside), "reasons": reasons,
                "samples": len(inside)}


class NvmlClocks:
    """Dense clock samples from NVML (read-only queries through ctypes): a
    thread polls the SM clock and the clock-event reasons every `period_s`
    while running.  Falls back to nothing (available False) when the NVML
    library cannot be loaded."""
    # nvmlClocksEventReasons bits of the public NVML API
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, device_index, period_s=0.0005):
        import ctypes
        import threading
        self.samples, self.available, self._stop = [], False, threading.Event()
        self.period = period_s
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                return
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
            h = ctypes.c_void_p()
            if nv.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(h)) != 0:
                return
            self._nv, self._h, self._ct = nv, h, ctypes
            mx = ctypes.c_uint(0)
            nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx))   # NVML_CLOCK_SM
            self.max_mhz = float(mx.value)
            self.available = True
        except Exception:
            return
        self._thread = threading.Thread(target=self._run, daemon=True)

    def _run(self):
        ct, nv, h = self._ct, self._nv, self._h
        mhz, rs = ct.c_uint(0), ct.c_ulonglong(0)
        while not self._stop.is_set():
            if nv.nvmlDeviceGetClockInfo(h, 1, ct.byref(mhz)) == 0:
                r = nv.nvmlDeviceGetCurrentClocksEventReasons(h, ct.byref(rs))
                self.samples.append((time.time(), float(mhz.value), rs.value if r == 0 else 0))
            time.sleep(self.period)

    def start(self):
        if self.available:
            self._thread.start()
        return self

    def stop(self):
        if self.available:
            self._stop.set()
            self._thread.join(timeout=5)

    def summary(self, t0, t1):
        if not self.available:
            return None
        inside = [s for s in self.samples if t0 <= s[0] <= t1]
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": ["no samples"],
                    "samples": 0, "source": "nvml"}
        reasons = sorted({n for _, _, r in inside for b, n in self.REASONS.items() if r & b})
        return {"sm_mhz": statistics.median(s[1] for s in inside), "sm_max_mhz": self.max_mhz,
                "sm_mhz_min": min(s[1] for s in inside), "reasons": reasons,
                "samples": len(inside), "source": "nvml, every 0.5 ms"}


# ------------------------------------------------------------- roofline ----

def env_info(dev):
    """The device and software a line was measured on (never raises)."""
    info = {"gpu": None, "sms": None, "cuda": torch.version.cuda, "torch": torch.__version__,
            "pkv_version": None}
    try:
        props = torch.cuda.get_device_properties(dev)
        info["gpu"], info["sms"] = props.name, props.multi_processor_count
    except Exception:
        pass
    try:
        import paged_kv_gqa_append_gb300 as pkv
        v = int(pkv.lib.pkv_version())
        info["pkv_version"] = f"{v // 10000}.{v // 100 % 100}.{v % 100}"
    except Exception:
        pass
    return info


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def ncu_traffic(kernel_tag):
    """dram bytes per launch recorded by ncu for this kernel source, else None."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    src = os.path.join(ROOT, "paged_kv_gqa_append_gb300", "csrc", "paged_decode.cu")
    try:
        sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
        for line in open(path):
            f = dict(kv.split("=", 1) for kv in line.split() if "=" in kv)
            if f.get("kernel") == kernel_tag and f.get("source_sha") == sha:
                return float(f["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


# ------------------------------------------------------------ CPU oracle ---

class OracleSample:
    """The FP64 oracle on one (layer, sequence) pair of the workload.

    One run: append the sequence's new token into its pages (K rotated, q
    rotated), then decode its 32 heads over the full context.
    """

    def __init__(self, case):
        from oracle import paged_kv as OP, rope as OR
        self.OP = OP
        self.case = case
        self.cos, self.sin = OR.table(OR.inv_freq_llama3(), W.MAX_CONTEXT)
        self.n = int(case.seq_lens[0])
        pages_per = (self.n + 15) // 16
        gen = W.cpu_gen(case.seed + 99)
        self.pool = W.bf16_bits(W.normal_bf16((pages_per, 2, 8, 16, 64), gen))
        self.bt = np.full((1, W.MAX_BLOCKS), -1, np.int32)
        self.bt[0, :pages_per] = np.arange(pages_per)
        self.k = W.bf16_bits(W.normal_bf16((1, 8, 64), gen))
        self.v = W.bf16_bits(W.normal_bf16((1, 8, 64), gen))
        self.q = W.bf16_bits(W.normal_bf16((1, 32, 64), gen))
        self.kv_bytes = self.n * W.NUM_KV_HEADS * W.HEAD_DIM * 2 * 2

    def run_one(self):
        p2, qr, _ = self.OP.append_rope(self.pool, self.k, self.v, np.array([self.n - 1]), None,
                                        self.bt, self.cos, self.sin, self.q)
        self.OP.decode(qr, p2, self.bt, np.array([self.n]), self.case.scale)

    def timed(self, budget_s):
        """Run pairs until budget_s has passed; returns (GB/s, pairs, seconds)."""
        done, t0 = 0, time.perf_counter()
        while True:
            self.run_one()
            done += 1
            el = time.perf_counter() - t0
            if el >= budget_s:
                return done * self.kv_bytes / el / 1e9, done, el


class OracleSampleInt8(OracleSample):
    """The same (layer, sequence) pair on INT8 pages: append the new token
    (K rotated and quantised, V quantised, q rotated), then decode."""

    def __init__(self, case):
        super().__init__(case)
        import dataclasses
        from oracle import int8_kv as OI
        self.OI = OI
        pages_per = self.pool.shape[0]
        small = dataclasses.replace(case, num_pages=pages_per, outlier_frac=0.0)
        self.codes, self.scales = OI.unpack_pages(W.fill_pool_int8(small).numpy())
        self.kv_bytes = self.n * W.NUM_KV_HEADS * INT8_ROW_BYTES

    def run_one(self):
        c2, s2, qr, _ = self.OI.append_rope_int8(self.codes, self.scales, self.k, self.v,
                                                 np.array([self.n - 1]), None, self.bt, self.cos,
                                                 self.sin, self.q)
        self.OI.decode_int8(qr, c2, s2, self.bt, np.array([self.n]), self.case.scale)


# K and V of one (token, KV head) on INT8 pages: 64 + 64 code bytes, 4 + 4 scale bytes
INT8_ROW_BYTES = 2 * (W.HEAD_DIM + 4)


def cpu_cores_used():
    return 1  # the oracle is single-threaded NumPy (BLAS pinned to one thread)


# ------------------------------------------------------------------- arms ---

def run_reference_other(args):
    """The oracle on the prefill or argmax workload (one bounded sample per step)."""
    if args.workload == "prefill":
        from oracle import paged_kv as OP
        pool_h, bt_h, q_h, _, lens_h = prefill_inputs(None)
        P, rows = PREFILL_P, 4
        q_s, cu_s, pool_bits = W.bf16_bits(q_h[P - rows:P]), np.array([0, rows], np.int32), W.bf16_bits(pool_h)
        one = lambda: OP.prefill(q_s, cu_s, pool_bits, bt_h[:1], lens_h[:1], W.DEFAULT_SCALE)
        work, unit, metric = rows * P * W.NUM_Q_HEADS * W.HEAD_DIM * 4 / 1e12, "TFLOP/s", \
            "paged causal prefill TFLOP/s (causal attention FLOPs)"
        sample = f"{rows} query rows at the end of a {P}-token prompt per step"
        workload = f"prefill_b{PREFILL_S}_p{P}"
    else:
        from oracle import argmax as OA
        x = torch.randn(ARGMAX_ROWS, ARGMAX_VOCAB, generator=torch.Generator().manual_seed(6)).numpy()
        one = lambda: OA.argmax_rows(x)
        work, unit, metric = ARGMAX_ROWS * ARGMAX_VOCAB * 4 / 1e9, "GB/s", \
            "next-token argmax GB/s (FP32 logits read)"
        sample = f"{ARGMAX_ROWS} rows of {ARGMAX_VOCAB} per step"
        workload = f"argmax_b{ARGMAX_ROWS}_v{ARGMAX_VOCAB}"
    for _ in range(args.warmup):
        one()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        one()
    el = time.perf_counter() - t0
    value = work * args.steps / el
    print(json.dumps({
        "impl": "reference", "metric": metric, "value": value, "unit": unit, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": workload, "sample": sample},
        "cpu_baseline": {"value": value, "unit": unit, "cores": cpu_cores_used(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}),
        flush=True)


def run_reference(args, world, rank):
    if rank != 0:
        return
    if args.workload in ("prefill", "argmax"):
        run_reference_other(args)
        return
    if args.workload == "continuous":
        from oracle import admission as OA
        case = W.case_continuous()
        _, log, _ = OA.simulate(case.prompt_lens, case.decode_steps, case.num_pages,
                                case.num_layers)
        tokens = sum(len(e["lens"]) for e in log)
        ora = mix_sample(round(sum(sum(e["lens"]) for e in log) / tokens))
        for _ in range(args.warmup):
            ora.run_one()
        t0 = time.perf_counter()
        for _ in range(args.steps):
            ora.run_one()
        el = time.perf_counter() - t0
        value = args.steps * ora.kv_bytes / el / 1e9
        sample = (f"{args.steps} (layer, sequence) pairs at the mix's mean decode length "
                  f"({ora.n} tokens): append 1 token + decode 32 heads each")
        print(json.dumps({
            "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": el / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": case.name, "requests": len(case.prompt_lens),
                       "layers": case.num_layers, "mean_len": ora.n,
                       "sample": "one (layer, seq) pair per step"},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cpu_cores_used(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}), flush=True)
        return
    if args.workload in ("mixed8", "single37"):
        from oracle import paged_kv as OP
        case = W.case_mixed() if args.workload == "mixed8" else W.case_single()
        pool_b = W.bf16_bits(W.fill_pool(case))
        q_b = W.bf16_bits(W.fill_queries(case))[0]
        one = lambda: OP.decode(q_b, pool_b, case.block_tables[0], case.seq_lens, case.scale)
        for _ in range(args.warmup):
            one()
        t0 = time.perf_counter()
        for _ in range(args.steps):
            one()
        el = time.perf_counter() - t0
        value = case.kv_bytes_per_layer() * args.steps / el / 1e9
        sample = f"{args.steps} whole decodes of {case.name}"
        print(json.dumps({
            "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": el / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": case.name, "batch": case.num_seqs, "layers": 1},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cpu_cores_used(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}), flush=True)
        return
    case = make_case(args.workload, args.layers)
    int8 = args.workload.startswith("int8")
    ora = OracleSampleInt8(case) if int8 else OracleSample(case)
    # warm-up steps, then K timed steps; each step = one (layer, seq) pair
    for _ in range(args.warmup):
        ora.run_one()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        ora.run_one()
    el = time.perf_counter() - t0
    pairs = args.steps
    n_tok = ora.n
    value = pairs * ora.kv_bytes / el / 1e9
    sample = (f"{pairs} (layer, sequence) pairs of {case.name}{' on INT8 pages' if int8 else ''}: "
              f"append 1 token + decode 32 heads over {n_tok} tokens each")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": el / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": ("int8_" if int8 else "") + case.name, "batch": case.num_seqs,
                   "layers": case.num_layers, "ctx": n_tok, "sample": "one (layer, seq) pair per step"},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cpu_cores_used(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_gb300(args, world, rank, local):
    import paged_kv_gqa_append_gb300 as pkv
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    case = make_case(args.workload, args.layers)
    L, S = case.num_layers, case.num_seqs
    compute = pkv.COMPUTE_TENSOR if args.compute == "tensor" else pkv.COMPUTE_FMA

    pool = W.fill_pool(case, device=dev)
    inbuf, (q_raw, k_new, v_new, pos, lens, bt) = packed_step_inputs(case, dev)
    cos, sin = pkv.rope_tables_device(dev, W.MAX_CONTEXT)
    out = torch.empty_like(q_raw)
    kv_bytes_layer = case.kv_bytes_per_layer()
    step = pkv.DecodeStep(pool, bt, lens, pos, k_new, v_new, q_raw, out, cos, sin, case.scale,
                          max_seq_len=case.max_seq_len,
                          compute=None if compute == pkv.COMPUTE_TENSOR else compute,
                          fused=not args.unfused,
                          schedule={"auto": 2, "static": 0, "dynamic": 1}[args.schedule])
    stream = torch.cuda.current_stream(dev)

    for _ in range(args.warmup):
        step.run()
    code = step.error()
    if code != 0:
        raise RuntimeError(f"device error {pkv.status_string(code)} during warm-up")

    # ---- headline: K graph replays of the step, inputs resident in HBM -----
    clocks = ClockSampler(dev.index) if rank == 0 else None
    dense = NvmlClocks(dev.index).start() if rank == 0 else None
    time.sleep(0.5 if clocks else 0)
    barrier(world)
    torch.cuda.synchronize()
    t_wall0 = time.time()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step.run()
    e1.record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    barrier(world)
    ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    # ---- the same step graph over a sustained window of >= 2 s, clocks sampled
    n_sus = 0 if args.no_sustained else max(1, int(2.0 / max(ms / args.steps / 1e3, 1e-6)) + 1)
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t_sus0 = time.time()
    s0.record(stream)
    for _ in range(n_sus):
        step.run()
    s1.record(stream)
    torch.cuda.synchronize()
    t_sus1 = time.time()
    sus_ms = s0.elapsed_time(s1)
    if dense:
        dense.stop()
    code = step.error()
    if code != 0:
        raise RuntimeError(f"device error {pkv.status_string(code)} in the timed region")

    # ---- roofline: the dominant kernel's average launch duration -----------
    if step.fused:
        # the step graph holds only the L fused decode-with-append launches,
        # so the headline region itself times that kernel
        k_roof = steps_timed = args.steps
        dec_avg_ms = ms / (steps_timed * L)
    else:
        g_dec = step.decode_only_graph()
        for _ in range(3):
            g_dec.replay()
        k_roof = max(10, args.steps // 4)
        r0, r1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        r0.record(stream)
        for _ in range(k_roof):
            g_dec.replay()
        r1.record(stream)
        torch.cuda.synchronize()
        dec_avg_ms = r0.elapsed_time(r1) / (k_roof * L)
    # ---- the append kernel alone (kv_append_rope of the step's tokens) -----
    g_app = step.append_only_graph()
    for _ in range(3):
        g_app.replay()
    k_app = max(10, args.steps // 4)
    p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    p0.record(stream)
    for _ in range(k_app):
        g_app.replay()
    p1.record(stream)
    torch.cuda.synchronize()
    append_us = p0.elapsed_time(p1) * 1e3 / (k_app * L)
    if step.error() != 0:
        raise RuntimeError("device error in the append timing")
    t_wall2 = time.time()
    clk = clocks.summary(t_wall0, t_wall2) if clocks else None
    if clocks:
        clocks.stop()
    if dense and dense.available:
        # the headline's own clocks come from the dense samples of its region
        clk = dict(dense.summary(t_wall0, t_wall1), smi=clk)
    sustained = None
    if rank == 0 and n_sus:
        sus_clk = dense.summary(t_sus0, t_sus1) if dense and dense.available else None
        sustained = {"steps": n_sus, "ms_per_step": sus_ms / n_sus,
                     "value": kv_bytes_layer * L * n_sus / (sus_ms / 1e3) / 1e9, "unit": "GB/s",
                     "window_s": sus_ms / 1e3, "clocks": sus_clk}
        if sus_clk and sus_clk.get("sm_mhz"):
            # time x clock: the step's cost in SM cycles, comparable across clocks
            sustained["us_x_mhz_per_layer"] = sus_ms * 1e3 / (n_sus * L) * sus_clk["sm_mhz"]

    steps = args.steps
    sec = ms / 1e3
    total_kv = kv_bytes_layer * L * steps * world
    value = total_kv / sec / 1e9
    tokens_per_s = S * steps * world / sec
    us_per_layer = ms * 1e3 / (steps * L)

    # ---- e2e: the same step with its inputs uploaded and output read back --
    e2e = None
    if not args.no_e2e:
        in_h = inbuf.cpu().pin_memory()      # q, new K/V, positions, lengths, tables
        out_h = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
        h2d = in_h.numel()
        d2h = out_h.numel() * out_h.element_size()
        k_e2e = max(1, min(steps, 500))
        barrier(world)
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0 = time.perf_counter()
        a.record(stream)
        for _ in range(k_e2e):
            inbuf.copy_(in_h, non_blocking=True)     # the step's inputs: one upload
            step.run()
            out_h.copy_(out, non_blocking=True)
        b.record(stream)
        torch.cuda.synchronize()
        host_s = time.perf_counter() - t0
        e2e_s = max_over_ranks(max(a.elapsed_time(b) / 1e3, host_s), world, dev)
        e2e = {"value": kv_bytes_layer * L * k_e2e * world / e2e_s / 1e9, "unit": "GB/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "steps": k_e2e, "tokens_per_s": S * k_e2e * world / e2e_s,
               "path": "DecodeStep graph replay; the step's inputs (q, new K/V, positions, "
                       "lengths, tables) uploaded as one pinned copy, the output read back"}
        if step.error() != 0:
            raise RuntimeError("device error in the e2e region")

    # ---- roofline of the dominant kernel -----------------------------------
    peak, peak_kind = hbm_peak()
    achieved = kv_bytes_layer / (dec_avg_ms / 1e3) / 1e9
    tag = ("paged_decode_append" if step.fused else
           "paged_decode_" + ("mma" if compute == pkv.COMPUTE_TENSOR else "fma"))
    if effective_schedule(args.schedule, case, dev) == "dynamic":
        tag += "_dyn"
    traffic = ncu_traffic(f"{tag}:{case.name}")
    roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
            "frac": achieved / peak, "traffic": traffic, "peak_source": peak_kind,
            "kernel": (f"{tag} (paged_gqa_decode_append: the step's only kernel, one launch "
                       "per layer, timed over the headline region)" if step.fused else
                       f"{tag} (paged_gqa_decode: decode-only graph, one launch per layer)"),
            "launches_timed": k_roof * L,
            "algorithmic_bytes_per_launch": kv_bytes_layer,
            "avg_launch_us": dec_avg_ms * 1e3}

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        gbs, pairs, el = OracleSample(case).timed(10.0)
        cpu = {"value": gbs, "unit": "GB/s", "cores": cpu_cores_used(), "kind": "oracle",
               "sample": f"{pairs} (layer, sequence) pairs of {case.name} (append 1 token + "
                         f"decode 32 heads over {int(case.seq_lens[0])} tokens), {el:.1f} s"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": steps,
            "warmup": args.warmup, "ms_per_step": ms / steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": case.name, "batch": S, "layers": L,
                       "ctx": int(case.seq_lens[0]), "pool_pages": case.num_pages,
                       "pool_bytes": case.num_pages * W.PAGE_ELEMS * 2,
                       "l2": "inputs larger than L2 (pool read per step exceeds 129 MB L2)",
                       "parallelism": f"replicas x{world}", "compute": args.compute,
                       "schedule": f"{args.schedule} ({effective_schedule(args.schedule, case, dev)})",
                       "launch": ("CUDA graph of the step: one fused append+decode kernel per layer"
                                  if step.fused else
                                  "CUDA graph of the step: append kernel + decode kernel per layer")},
            "tokens_per_s": tokens_per_s, "us_per_layer": us_per_layer,
            "append_us_per_layer": append_us,
            "kv_bytes_per_step": kv_bytes_layer * L,
            "hbm_frac_step": value / world / peak,
            "clocks": clk, "sustained": sustained, "e2e": e2e,
            "gpu_launches": step.launches_per_step * steps,
            "roofline": roof, "env": env_info(dev), "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)


def packed_step_inputs(case, dev):
    """The step's inputs (q, new K/V, positions, lengths, tables) as views of
    one device buffer, so that an end-to-end run uploads them in one copy.
    Returns (buffer, [q, k_new, v_new, positions, lengths, tables])."""
    parts = [W.fill_queries(case, device=dev), *W.fill_new_kv(case, device=dev),
             torch.from_numpy(W.new_positions(case)).to(dev),
             torch.from_numpy(case.seq_lens).to(dev), torch.from_numpy(case.block_tables).to(dev)]
    offs, total = [], 0
    for x in parts:
        offs.append(total)
        total += (x.numel() * x.element_size() + 255) // 256 * 256
    inbuf = torch.empty(total, dtype=torch.uint8, device=dev)
    views = []
    for x, o in zip(parts, offs):
        v = inbuf[o:o + x.numel() * x.element_size()].view(x.dtype).view(x.shape)
        v.copy_(x)
        views.append(v)
    return inbuf, views


# ---------------------------------------------------------- INT8 pages ----

def run_int8_line(args, world, rank, local):
    """The decode step on INT8 K/V pages: per layer one fused kernel
    (paged_gqa_decode_append_int8: new token quantised into its page, q
    rotated, attention), or with --unfused kv_append_rope_int8 then
    paged_gqa_decode_int8; one CUDA graph per step.  KV bytes per (token,
    head): 136 (codes and scales)."""
    import paged_kv_gqa_append_gb300 as pkv
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    case = make_case(args.workload, args.layers)
    L, S = case.num_layers, case.num_seqs
    pool = W.fill_pool_int8(case, device=dev)
    inbuf, (q_raw, k_new, v_new, pos, lens, bt) = packed_step_inputs(case, dev)
    cos, sin = pkv.rope_tables_device(dev, W.MAX_CONTEXT)
    out = torch.empty_like(q_raw)
    kv_bytes_layer = int(case.seq_lens.sum()) * W.NUM_KV_HEADS * INT8_ROW_BYTES
    step = pkv.Int8DecodeStep(pool, bt, lens, pos, k_new, v_new, q_raw, out, cos, sin,
                              case.scale, max_seq_len=case.max_seq_len,
                              fused=False if args.unfused else None)   # None: the fused kernel
    stream = torch.cuda.current_stream(dev)
    for _ in range(args.warmup):
        step.run()
    if step.error() != 0:
        raise RuntimeError("device error during the INT8 warm-up")

    def timed(run, k):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record(stream)
        for _ in range(k):
            run()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b)

    clocks = ClockSampler(dev.index) if rank == 0 else None
    time.sleep(0.5 if clocks else 0)
    barrier(world)
    t_wall0 = time.time()
    ms = max_over_ranks(timed(step.run, args.steps), world, dev)
    barrier(world)
    if step.error() != 0:
        raise RuntimeError("device error in the INT8 timed region")
    # the dominant kernel: the fused kernel is the step's only kernel (timed
    # over the headline region); else the decode kernel alone.  And the
    # append kernel alone.
    g_dec, g_app = step.partial_graph(False, True), step.partial_graph(True, False)
    for _ in range(3):
        g_dec.replay()
        g_app.replay()
    k_part = max(10, args.steps // 4)
    dec_only_ms = timed(g_dec.replay, k_part) / (k_part * L)
    dec_avg_ms = ms / (args.steps * L) if step.fused else dec_only_ms
    append_us = timed(g_app.replay, k_part) * 1e3 / (k_part * L)
    if step.error() != 0:
        raise RuntimeError("device error in the INT8 kernel timings")
    clk = clocks.summary(t_wall0, time.time()) if clocks else None
    if clocks:
        clocks.stop()
    steps = args.steps
    sec = ms / 1e3
    value = kv_bytes_layer * L * steps * world / sec / 1e9

    e2e = None
    if not args.no_e2e:
        in_h = inbuf.cpu().pin_memory()      # q, new K/V, positions, lengths, tables
        out_h = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
        h2d = in_h.numel()
        k_e2e = max(1, min(steps, 500))

        def e2e_step():
            inbuf.copy_(in_h, non_blocking=True)     # the step's inputs: one upload
            step.run()
            out_h.copy_(out, non_blocking=True)
        barrier(world)
        t0 = time.perf_counter()
        dev_ms = timed(e2e_step, k_e2e)
        e2e_s = max_over_ranks(max(dev_ms / 1e3, time.perf_counter() - t0), world, dev)
        e2e = {"value": kv_bytes_layer * L * k_e2e * world / e2e_s / 1e9, "unit": "GB/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": out_h.numel() * out_h.element_size(),
               "steps": k_e2e, "tokens_per_s": S * k_e2e * world / e2e_s,
               "path": "Int8DecodeStep graph replay; the step's inputs (q, new K/V, positions, "
                       "lengths, tables) uploaded as one pinned copy, the output read back"}
        if step.error() != 0:
            raise RuntimeError("device error in the INT8 e2e region")

    peak, peak_kind = hbm_peak()
    achieved = kv_bytes_layer / (dec_avg_ms / 1e3) / 1e9
    tag = "paged_decode_append_int8" if step.fused else "paged_decode_int8"
    roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
            "frac": achieved / peak, "traffic": ncu_traffic(f"{tag}:{case.name}"),
            "peak_source": peak_kind,
            "kernel": (f"{tag} (paged_gqa_decode_append_int8: the step's only kernel, one launch "
                       "per layer, timed over the headline region)" if step.fused else
                       f"{tag} (paged_gqa_decode_int8: decode-only graph, one launch per layer)"),
            "launches_timed": (args.steps if step.fused else k_part) * L,
            "algorithmic_bytes_per_launch": kv_bytes_layer,
            "avg_launch_us": dec_avg_ms * 1e3}
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        gbs, pairs, el = OracleSampleInt8(case).timed(10.0)
        cpu = {"value": gbs, "unit": "GB/s", "cores": cpu_cores_used(), "kind": "oracle",
               "sample": f"{pairs} (layer, sequence) pairs of {case.name} on INT8 pages (append "
                         f"1 token + decode 32 heads over {int(case.seq_lens[0])} tokens), {el:.1f} s"}
    if rank == 0:
        print(json.dumps({
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": steps,
            "warmup": args.warmup, "ms_per_step": ms / steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "int8",
            "data": "synthetic",
            "config": {"workload": "int8_" + case.name, "batch": S, "layers": L,
                       "ctx": int(case.seq_lens[0]), "pool_pages": case.num_pages,
                       "pool_bytes": case.num_pages * W.NUM_KV_HEADS * W.I8_BLOCK_BYTES,
                       "kv_format": "int8 codes + fp32 scale per (token, KV head) row of K and V, "
                                    "one 2176-byte block per (page, KV head); fp16 tensor-core "
                                    "MMAs, fp32 accumulation",
                       "l2": "inputs larger than L2 (pool read per step exceeds 129 MB L2)",
                       "parallelism": f"replicas x{world}",
                       "launch": ("CUDA graph of the step: one fused INT8 append+decode kernel per layer"
                                  if step.fused else
                                  "CUDA graph of the step: INT8 append kernel + INT8 decode kernel per layer")},
            "tokens_per_s": S * steps * world / sec, "us_per_layer": ms * 1e3 / (steps * L),
            "decode_only_us_per_layer": dec_only_ms * 1e3, "append_us_per_layer": append_us,
            "kv_bytes_per_step": kv_bytes_layer * L, "hbm_frac_step": value / world / peak,
            "clocks": clk, "e2e": e2e, "gpu_launches": step.launches_per_step * steps,
            "roofline": roof, "env": env_info(dev), "cpu_baseline": cpu}), flush=True)


# ------------------------------------------- the small decode cases ------

def run_small_line(args, world, rank, local):
    """One paged_gqa_decode launch on a small case: the batch of 8 mixed
    lengths (16.8 MB of K/V, which fits in L2: timed with a 2 x L2 buffer
    written before each launch, and warm, back to back, beside it) or the one
    37-token sequence (latency: microseconds per call)."""
    import paged_kv_gqa_append_gb300 as pkv
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    case = W.case_mixed() if args.workload == "mixed8" else W.case_single()
    pool = W.fill_pool(case, device=dev)
    q = W.fill_queries(case, device=dev)[0]
    bt = torch.from_numpy(case.block_tables[0]).to(dev)
    lens = torch.from_numpy(case.seq_lens).to(dev)
    out = torch.empty_like(q)
    ws = pkv.alloc_workspace(case.num_seqs, dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    kv_bytes = case.kv_bytes_per_layer()
    stream = torch.cuda.current_stream(dev)
    launch = lambda: pkv.paged_gqa_decode(q, pool, bt, lens, out, case.scale, workspace=ws,
                                          max_seq_len=case.max_seq_len, d_err=err)
    launch()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        launch()
    for _ in range(max(3, args.warmup)):
        g.replay()
    if pkv.pkv_read_device_error(err):
        raise RuntimeError("device error in the warm-up")
    steps = max(1, min(args.steps, 500))
    flush = torch.empty(2 * 129 * 2 ** 20 // 4, dtype=torch.float32, device=dev)  # 2 x L2
    clocks = ClockSampler(dev.index) if rank == 0 else None
    time.sleep(0.5 if clocks else 0)
    barrier(world)
    torch.cuda.synchronize()
    t_wall0 = time.time()
    # flushed: events around each launch, the L2 flush outside them
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    for a, b in evs:
        flush.fill_(1.0)
        a.record(stream)
        g.replay()
        b.record(stream)
    torch.cuda.synchronize()
    flushed_ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in evs), world, dev)
    # warm: back to back
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        g.replay()
    b.record(stream)
    torch.cuda.synchronize()
    warm_ms = max_over_ranks(a.elapsed_time(b), world, dev)
    clk = clocks.summary(t_wall0, time.time()) if clocks else None
    if clocks:
        clocks.stop()
    if pkv.pkv_read_device_error(err):
        raise RuntimeError("device error in the timed region")
    us_flushed, us_warm = flushed_ms * 1e3 / steps, warm_ms * 1e3 / steps
    value = kv_bytes * steps * world / (flushed_ms / 1e3) / 1e9
    # e2e: q uploaded from pinned memory, the output read back, per launch
    q_h, out_h = q.cpu().pin_memory(), torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    k_e2e = max(1, min(steps, 200))
    torch.cuda.synchronize()
    a.record(stream)
    t0 = time.perf_counter()
    for _ in range(k_e2e):
        q.copy_(q_h, non_blocking=True)
        g.replay()
        out_h.copy_(out, non_blocking=True)
    b.record(stream)
    torch.cuda.synchronize()
    e2e_s = max_over_ranks(max(a.elapsed_time(b) / 1e3, time.perf_counter() - t0), world, dev)
    peak, peak_kind = hbm_peak()
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        from oracle import paged_kv as OP
        pool_b, q_b = W.bf16_bits(pool), W.bf16_bits(q)
        done, t0 = 0, time.perf_counter()
        while time.perf_counter() - t0 < 5.0:
            OP.decode(q_b, pool_b, case.block_tables[0], case.seq_lens, case.scale)
            done += 1
        el = time.perf_counter() - t0
        cpu = {"value": kv_bytes * done / el / 1e9, "unit": "GB/s", "cores": cpu_cores_used(),
               "kind": "oracle", "sample": f"{done} whole decodes of {case.name}, {el:.1f} s"}
    if rank == 0:
        print(json.dumps({
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": steps,
            "warmup": args.warmup, "ms_per_step": flushed_ms / steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": case.name, "batch": case.num_seqs, "layers": 1,
                       "seq_lens": [int(x) for x in case.seq_lens], "pool_pages": case.num_pages,
                       "l2": "flushed: a 2 x L2 buffer written before each timed launch (outside "
                             "its events); `warm_us_per_call` times back-to-back launches",
                       "parallelism": f"replicas x{world}",
                       "launch": "one paged_gqa_decode launch (CUDA graph replay) per step"},
            "us_per_call": us_flushed, "warm_us_per_call": us_warm,
            "warm_gbs": kv_bytes * steps * world / (warm_ms / 1e3) / 1e9,
            "kv_bytes_per_step": kv_bytes, "clocks": clk, "gpu_launches": steps,
            "e2e": {"value": kv_bytes * k_e2e * world / e2e_s / 1e9, "unit": "GB/s",
                    "h2d_bytes_per_step": q_h.numel() * 2, "d2h_bytes_per_step": out_h.numel() * 2,
                    "steps": k_e2e},
            "roofline": {"bound": "hbm", "achieved": value / world, "peak": peak, "unit": "GB/s",
                         "frac": value / world / peak, "traffic": None, "peak_source": peak_kind,
                         "kernel": "paged_decode_kernel (paged_gqa_decode, L2 flushed before each launch)",
                         "avg_launch_us": us_flushed, "algorithmic_bytes_per_launch": kv_bytes},
            "env": env_info(dev), "cpu_baseline": cpu}), flush=True)


# ------------------------------------------------ continuous-batching line --

SLEEP_CYCLES = 20_000_000  # ~10 ms at 2 GHz: covers the host's enqueue of one step


def mix_sample(mean_len):
    """The oracle on one (layer, sequence) pair at the mix's mean decode length."""
    n = int(mean_len)
    case = W.DecodeCase("continuous_r64_geo300", 3, 16, np.array([n], np.int32), 0,
                        np.zeros((1, 1, W.MAX_BLOCKS), np.int32))
    return OracleSample(case)


def run_continuous_line(args, world, rank, local):
    """The continuous-batching mix run to completion through
    serving.ContinuousBatcher: 64 requests (prompts geometric, mean 300,
    clipped to [1, 1920]) of 128 decode steps each, 16 layers, a 128 MiB pool
    of 4096 pages, admission by page credit, one fused append + decode kernel
    per layer and step.

    Device time: each step's host work (scheduler, table rows, the batch's
    table gather, that step's q / k / v drawn on the device) is queued first,
    then a 2 x L2 buffer is written and a device sleep queued so that the
    step's 16 launches are all queued before the GPU reaches them; CUDA
    events bracket those launches alone.  (The host's enqueue time also
    counts waits on a full launch queue, when it has run ahead of the
    device; the measured step times were the same with a 3 ms sleep.)  value = K/V bytes the steps read
    (sum over steps, layers and sequences of length x 2048) / the summed step
    time.  e2e: the same mix again, wall clock from the first admission to
    the last output read back, prompts and every step's q / k / v copied from
    pinned host memory and every step's output copied to pinned host memory.
    """
    import paged_kv_gqa_append_gb300 as pkv
    from paged_kv_gqa_append_gb300.serving import ContinuousBatcher
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    case = W.case_continuous()
    L = case.num_layers
    cos, sin = pkv.rope_tables_device(dev, W.MAX_CONTEXT)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(2 * 129 * 2 ** 20 // 4, dtype=torch.float32, device=dev)  # 2 x L2
    gen = torch.Generator(device=dev)
    gen.manual_seed(case.seed)
    pmax = int(case.prompt_lens.max())
    prompt_d = W.normal_bf16((2, pmax, W.NUM_KV_HEADS, W.HEAD_DIM), gen)

    def batcher():
        pool = torch.zeros((case.num_pages, 2, 8, 16, 64), dtype=torch.bfloat16, device=dev)
        cb = ContinuousBatcher(pool, L, cos, sin, W.DEFAULT_SCALE, max_slots=64)
        for p in case.prompt_lens:
            if cb.submit(int(p), case.allowed_new_tokens) < 0:
                raise RuntimeError("request rejected")
        return cb

    def device_run(max_steps):
        cb = batcher()
        P = lambda rid, l: (prompt_d[0, :cb.prompt[rid]], prompt_d[1, :cb.prompt[rid]])
        evs, host_s, tokens, kv_bytes, step = [], [], 0, 0, 0
        while (cb.sched.stats()["queued"] or cb.running) and step < max_steps:
            cb.admit(P)
            batch = cb.prepare_step()
            B = len(batch.ids)
            q = W.normal_bf16((L, B, W.NUM_Q_HEADS, W.HEAD_DIM), gen)
            k = W.normal_bf16((L, B, W.NUM_KV_HEADS, W.HEAD_DIM), gen)
            v = W.normal_bf16((L, B, W.NUM_KV_HEADS, W.HEAD_DIM), gen)
            flush.fill_(1.0)
            e0, e1, e2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
            e0.record(stream)
            torch.cuda._sleep(SLEEP_CYCLES)
            t0 = time.perf_counter()
            e1.record(stream)
            cb.launch_step(batch, q, k, v)
            e2.record(stream)
            host_s.append(time.perf_counter() - t0)
            evs.append((e0, e1, e2))
            tokens += B
            kv_bytes += int(batch.lens_h.sum()) * W.NUM_KV_HEADS * W.HEAD_DIM * 2 * 2 * L
            cb.retire(case.decode_steps)
            step += 1
        torch.cuda.synchronize()
        if cb.error():
            raise RuntimeError("device error in the continuous mix")
        step_ms = [a.elapsed_time(b) for _, a, b in evs]
        sleep_ms = [s.elapsed_time(a) for s, a, _ in evs]
        return step, tokens, kv_bytes, step_ms, sleep_ms, host_s

    def e2e_run():
        cb = batcher()
        bmax = 64
        prompt_h = prompt_d.cpu().pin_memory()
        # a step's q, k and v packed in one pinned block: one upload per step
        qkv_h = W.normal_bf16((L * bmax * (W.NUM_Q_HEADS + 2 * W.NUM_KV_HEADS) * W.HEAD_DIM,),
                              gen).cpu().pin_memory()
        out_h = torch.empty(L * bmax * W.NUM_Q_HEADS * W.HEAD_DIM, dtype=torch.bfloat16,
                            pin_memory=True)
        P = lambda rid, l: (prompt_h[0, :cb.prompt[rid]], prompt_h[1, :cb.prompt[rid]])
        h2d = d2h = steps = 0
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        while cb.sched.stats()["queued"] or cb.running:
            for rid in cb.admit(P):
                h2d += 2 * L * cb.prompt[rid] * W.NUM_KV_HEADS * W.HEAD_DIM * 2
            batch = cb.prepare_step()
            B = len(batch.ids)
            nq, nkv = L * B * W.NUM_Q_HEADS * W.HEAD_DIM, L * B * W.NUM_KV_HEADS * W.HEAD_DIM
            qkv = qkv_h[:nq + 2 * nkv].to(dev, non_blocking=True)
            q = qkv[:nq].view(L, B, W.NUM_Q_HEADS, W.HEAD_DIM)
            k = qkv[nq:nq + nkv].view(L, B, W.NUM_KV_HEADS, W.HEAD_DIM)
            v = qkv[nq + nkv:].view(L, B, W.NUM_KV_HEADS, W.HEAD_DIM)
            out = cb.launch_step(batch, q, k, v)
            out_h[:nq].copy_(out.view(-1), non_blocking=True)
            h2d += (nq + 2 * nkv) * 2
            d2h += nq * 2
            cb.retire(case.decode_steps)
            steps += 1
        torch.cuda.synchronize()
        el = time.perf_counter() - t0
        if cb.error():
            raise RuntimeError("device error in the continuous mix (e2e)")
        return el, steps, h2d + cb.uploaded_bytes, d2h

    device_run(max(3, args.warmup))          # warm-up: the first steps of the mix
    clocks = ClockSampler(dev.index) if rank == 0 else None
    time.sleep(0.5 if clocks else 0)
    barrier(world)
    torch.cuda.synchronize()
    t_wall0 = time.time()
    steps, tokens, kv_bytes, step_ms, sleep_ms, host_s = device_run(1 << 30)
    clk = clocks.summary(t_wall0, time.time()) if clocks else None
    if clocks:
        clocks.stop()
    total_ms = max_over_ranks(sum(step_ms), world, dev)
    value = kv_bytes * world / (total_ms / 1e3) / 1e9
    e2e_s, e2e_steps, h2d, d2h = e2e_run()
    if e2e_steps != steps:
        raise RuntimeError("the e2e run took another schedule")
    e2e_s = max_over_ranks(e2e_s, world, dev)
    peak, peak_kind = hbm_peak()
    mean_len = kv_bytes / (tokens * W.NUM_KV_HEADS * W.HEAD_DIM * 4 * L)
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        ora = mix_sample(round(mean_len))
        gbs, done, el = ora.timed(10.0)
        cpu = {"value": gbs, "unit": "GB/s", "cores": cpu_cores_used(), "kind": "oracle",
               "sample": f"{done} (layer, sequence) pairs at the mix's mean decode length "
                         f"({ora.n} tokens): append 1 token + decode 32 heads, {el:.1f} s"}
    if rank == 0:
        print(json.dumps({
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": steps,
            "warmup": max(3, args.warmup), "ms_per_step": total_ms / steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": case.name, "requests": len(case.prompt_lens),
                       "decode_steps_per_request": case.decode_steps, "layers": L,
                       "pool_pages": case.num_pages, "mean_batch": tokens / steps,
                       "mean_len": mean_len,
                       "l2": "flushed: a 2 x L2 buffer written before each step (outside its events)",
                       "parallelism": f"replicas x{world}",
                       "launch": "ContinuousBatcher.launch_step: one fused append+decode kernel "
                                 "per layer; events around each step's launches"},
            "tokens_per_s": tokens * world / (total_ms / 1e3),
            "us_per_layer": total_ms * 1e3 / (steps * L),
            "kv_bytes_total": kv_bytes,
            "host_enqueue_us_max": max(host_s) * 1e6,
            "host_enqueue_us_mean": sum(host_s) / len(host_s) * 1e6,
            "device_sleep_us_min": min(sleep_ms) * 1e3,
            "clocks": clk, "gpu_launches": steps * L,
            "e2e": {"value": kv_bytes * world / e2e_s / 1e9, "unit": "GB/s",
                    "h2d_bytes_per_step": h2d // e2e_steps, "d2h_bytes_per_step": d2h // e2e_steps,
                    "steps": e2e_steps, "tokens_per_s": tokens * world / e2e_s,
                    "path": "ContinuousBatcher admit / prepare_step / launch_step / retire, "
                            "inputs from and outputs to pinned host memory, host scheduling "
                            "included"},
            "roofline": {"bound": "hbm", "achieved": value / world, "peak": peak, "unit": "GB/s",
                         "frac": value / world / peak, "traffic": None, "peak_source": peak_kind,
                         "kernel": "paged_decode_append (one launch per layer and step)",
                         "launches_timed": steps * L, "avg_launch_us": total_ms * 1e3 / (steps * L),
                         "algorithmic_bytes_per_launch": kv_bytes / (steps * L)},
            "env": env_info(dev), "cpu_baseline": cpu}), flush=True)


# ------------------------------------------------ prefill and argmax lines --

def tensor_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "measured (bf16 burst)"
    except Exception:
        return FALLBACK_BF16_TFLOPS, "fallback"


PREFILL_S, PREFILL_P = 8, 1920   # prompts x tokens (the longest prompts of the mix)


def prefill_flops(S, P):
    """Causal attention FLOPs: sum over queries of (keys seen) x 32 heads x 64 x 4."""
    return S * (P * (P + 1) // 2) * W.NUM_Q_HEADS * W.HEAD_DIM * 4


def prefill_inputs(dev):
    S, P = PREFILL_S, PREFILL_P
    pages_per = (P + W.PAGE_TOKENS - 1) // W.PAGE_TOKENS
    num_pages = S * pages_per
    gen = W.cpu_gen(5)
    pool = W.normal_bf16((num_pages, 2, 8, 16, 64), gen)
    perm = np.random.default_rng(5).permutation(num_pages).astype(np.int32)
    bt = np.full((S, W.MAX_BLOCKS), -1, np.int32)
    for s in range(S):
        bt[s, :pages_per] = perm[s * pages_per:(s + 1) * pages_per]
    q = W.normal_bf16((S * P, W.NUM_Q_HEADS, W.HEAD_DIM), gen)
    cu = np.arange(0, S * P + 1, P, dtype=np.int32)
    lens = np.full(S, P, np.int32)
    return pool, bt, q, cu, lens


def run_prefill_line(args, world, rank, local):
    import paged_kv_gqa_append_gb300 as pkv
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    S, P = PREFILL_S, PREFILL_P
    pool_h, bt_h, q_h, cu_h, lens_h = prefill_inputs(dev)
    pool, q = pool_h.to(dev), q_h.to(dev)
    bt, cu, lens = (torch.from_numpy(a).to(dev) for a in (bt_h, cu_h, lens_h))
    out = torch.empty_like(q)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    run = lambda: pkv.paged_gqa_prefill(q, cu, pool, bt, lens, out, W.DEFAULT_SCALE, max_q_len=P,
                                        d_err=err)
    for _ in range(args.warmup):
        run()
    if pkv.pkv_read_device_error(err):
        raise RuntimeError("device error in prefill warm-up")
    steps = max(1, min(args.steps, 200))
    clocks = ClockSampler(dev.index) if rank == 0 else None
    time.sleep(0.5 if clocks else 0)
    barrier(world)
    torch.cuda.synchronize()
    t_wall0 = time.time()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        run()
    e1.record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    clk = clocks.summary(t_wall0, t_wall1) if clocks else None
    if clocks:
        clocks.stop()
    if pkv.pkv_read_device_error(err):
        raise RuntimeError("device error in the prefill timed region")
    flops = prefill_flops(S, P)
    value = flops * steps * world / (ms / 1e3) / 1e12
    # e2e: q uploaded from pinned memory and out read back every step
    q_pin, out_pin = q_h.pin_memory(), torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    k_e2e = max(1, min(steps, 50))
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.perf_counter()
    a.record(stream)
    for _ in range(k_e2e):
        q.copy_(q_pin, non_blocking=True)
        run()
        out_pin.copy_(out, non_blocking=True)
    b.record(stream)
    torch.cuda.synchronize()
    e2e_s = max_over_ranks(max(a.elapsed_time(b) / 1e3, time.perf_counter() - t0), world, dev)
    peak, kind = tensor_peak()
    avg_us = ms * 1e3 / steps
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        from oracle import paged_kv as OP
        rows = 4   # the last 4 queries of the first prompt (each sees ~1920 keys)
        q_s = W.bf16_bits(q_h[P - rows:P])
        cu_s = np.array([0, rows], np.int32)
        pool_bits = W.bf16_bits(pool_h)
        done, t0 = 0, time.perf_counter()
        while time.perf_counter() - t0 < 10.0:
            OP.prefill(q_s, cu_s, pool_bits, bt_h[:1], lens_h[:1], W.DEFAULT_SCALE)
            done += 1
        el = time.perf_counter() - t0
        cpu_flops = done * rows * P * W.NUM_Q_HEADS * W.HEAD_DIM * 4
        cpu = {"value": cpu_flops / el / 1e12, "unit": "TFLOP/s", "cores": cpu_cores_used(),
               "kind": "oracle", "sample": f"{done} x {rows} query rows at positions "
                                           f"{P - rows}..{P - 1} of a {P}-token prompt, {el:.1f} s"}
    if rank == 0:
        print(json.dumps({
            "metric": "paged causal prefill TFLOP/s (causal attention FLOPs)", "value": value,
            "unit": "TFLOP/s", "n_gpus": world, "steps": steps, "warmup": args.warmup,
            "ms_per_step": ms / steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": f"prefill_b{S}_p{P}", "prompts": S, "prompt_tokens": P,
                       "l2": "q (63 MB), out (63 MB) and pool (31.5 MB) together exceed the 129 MB L2; each page is read by up to 60 query blocks",
                       "parallelism": f"replicas x{world}"},
            "clocks": clk, "gpu_launches": steps,
            "e2e": {"value": flops * k_e2e * world / e2e_s / 1e12, "unit": "TFLOP/s",
                    "h2d_bytes_per_step": q_pin.numel() * 2, "d2h_bytes_per_step": out_pin.numel() * 2,
                    "steps": k_e2e},
            "roofline": {"bound": "tensor", "achieved": value / world, "peak": peak,
                         "unit": "TFLOP/s", "frac": value / world / peak, "traffic": None,
                         "peak_source": kind, "kernel": "paged_prefill_tc_kernel (tcgen05 bf16, S and O in tensor memory)",
                         "avg_launch_us": avg_us, "algorithmic_flops_per_launch": flops},
            "env": env_info(dev), "cpu_baseline": cpu}), flush=True)


ARGMAX_ROWS, ARGMAX_VOCAB, ARGMAX_BUFS = 32, 128256, 12   # 12 x 16.4 MB > L2


def run_argmax_line(args, world, rank, local):
    import paged_kv_gqa_append_gb300 as pkv
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    gen = torch.Generator().manual_seed(6)
    host = [torch.randn(ARGMAX_ROWS, ARGMAX_VOCAB, generator=gen) for _ in range(ARGMAX_BUFS)]
    bufs = [h.to(dev) for h in host]
    out = torch.empty(ARGMAX_ROWS, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    for i in range(max(args.warmup, 3)):
        pkv.argmax_rows(bufs[i % ARGMAX_BUFS], out)
    steps = max(ARGMAX_BUFS, min(args.steps, 2000))
    torch.cuda.synchronize()
    clocks = ClockSampler(dev.index) if rank == 0 else None
    time.sleep(0.5 if clocks else 0)
    barrier(world)
    t_wall0 = time.time()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(steps):
        pkv.argmax_rows(bufs[i % ARGMAX_BUFS], out)   # inputs rotate through > L2 of buffers
    e1.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    clk = clocks.summary(t_wall0, time.time()) if clocks else None
    if clocks:
        clocks.stop()
    nbytes = ARGMAX_ROWS * ARGMAX_VOCAB * 4
    value = nbytes * steps * world / (ms / 1e3) / 1e9
    peak, kind = hbm_peak()
    # e2e: logits uploaded from pinned memory, ids read back, every step
    pin = host[0].pin_memory()
    ids = torch.empty(ARGMAX_ROWS, dtype=torch.int32, pin_memory=True)
    k_e2e = 200
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.perf_counter()
    a.record(stream)
    for _ in range(k_e2e):
        bufs[0].copy_(pin, non_blocking=True)
        pkv.argmax_rows(bufs[0], out)
        ids.copy_(out, non_blocking=True)
    b.record(stream)
    torch.cuda.synchronize()
    e2e_s = max_over_ranks(max(a.elapsed_time(b) / 1e3, time.perf_counter() - t0), world, dev)
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        from oracle import argmax as OA
        x = host[0].numpy()
        done, t0 = 0, time.perf_counter()
        while time.perf_counter() - t0 < 5.0:
            OA.argmax_rows(x)
            done += 1
        el = time.perf_counter() - t0
        cpu = {"value": nbytes * done / el / 1e9, "unit": "GB/s", "cores": cpu_cores_used(),
               "kind": "oracle", "sample": f"{done} x {ARGMAX_ROWS} rows of {ARGMAX_VOCAB}, {el:.1f} s"}
    if rank == 0:
        print(json.dumps({
            "metric": "next-token argmax GB/s (FP32 logits read)", "value": value, "unit": "GB/s",
            "n_gpus": world, "steps": steps, "warmup": args.warmup, "ms_per_step": ms / steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": {"workload": f"argmax_b{ARGMAX_ROWS}_v{ARGMAX_VOCAB}", "rows": ARGMAX_ROWS,
                       "vocab": ARGMAX_VOCAB,
                       "l2": f"{ARGMAX_BUFS} input buffers rotated, {ARGMAX_BUFS * nbytes >> 20} MiB > L2",
                       "parallelism": f"replicas x{world}"},
            "us_per_step": ms * 1e3 / steps, "clocks": clk, "gpu_launches": steps,
            "e2e": {"value": nbytes * k_e2e * world / e2e_s / 1e9, "unit": "GB/s",
                    "h2d_bytes_per_step": nbytes, "d2h_bytes_per_step": ARGMAX_ROWS * 4,
                    "steps": k_e2e},
            "roofline": {"bound": "hbm", "achieved": value / world, "peak": peak, "unit": "GB/s",
                         "frac": value / world / peak, "traffic": None, "peak_source": kind,
                         "kernel": "argmax_kernel", "avg_launch_us": ms * 1e3 / steps,
                         "algorithmic_bytes_per_launch": nbytes},
            "env": env_info(dev), "cpu_baseline": cpu}), flush=True)


def main():
    args = parse()
    world, rank, local = dist_setup(args.gpus)
    try:
        if args.impl == "reference":
            run_reference(args, world, rank)
        elif args.workload == "prefill":
            run_prefill_line(args, world, rank, local)
        elif args.workload == "argmax":
            run_argmax_line(args, world, rank, local)
        elif args.workload.startswith("int8"):
            run_int8_line(args, world, rank, local)
        elif args.workload in ("mixed8", "single37"):
            run_small_line(args, world, rank, local)
        elif args.workload == "continuous":
            run_continuous_line(args, world, rank, local)
        else:
            run_gb300(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
