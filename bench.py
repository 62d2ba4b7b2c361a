"""Benchmark of the fused GEMM-epilogue / B2BGEMM path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one call of the fused kernel over one batch of synthetic inputs
that are already resident in HBM; L2 is flushed (a 256 MB write) between
timed steps.  The default workload, the one on the top level of the line, is
the largest configuration: the attention-shaped B2BGEMM (32 x 16 heads,
L = 2048, d = 128, softmax).  The line's ``configs`` object carries every
other configuration of the metric measured in the same run (GEMM + bias +
LayerNorm 256^3, GEMM + bias + tanh-GELU + RMSNorm 8192x4096x4096, the
scaled-softmax logit head 4096x16384x4096, the MLP B2BGEMM and the ReLU
attention variant), each with the same fields.  Rank 0 prints ONE JSON line.

``--impl reference`` times the float64 CPU oracle (the reference arm of this
build, a deliberately slow plain implementation) on the host cores instead.
Under torchrun (N > 1) every rank runs an independent replica of the
workload (rows are independent problems; no collective on the data path).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from back_gemm_fusion_gb300 import inputs as I  # noqa: E402

METRIC = "fused TFLOP/s & % of GB300 roofline; intermediate HBM bytes (target 0)"

# DRAM traffic of one fused launch (dram__bytes_read.sum, dram__bytes_write.sum)
# from `ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum,... -k <fused
# kernel> -c 1 bench.py --workload W --once` on a GB300 (fp32 output), keyed
# by workload; valid only while the hash of the workload's kernel family
# sources (kernel_source_hash) matches the one the counters were taken with,
# and for the workloads sized by --rows only at the rows they were taken at
# (profiles/ has the summaries and commands).
NCU_TRAFFIC = {
    "attention_long_keys": {"read": 67437568, "write": 290560, "src": "2be13edd6b10da33"},
    "attention_relu": {"read": 805388800, "write": 502074880, "src": "2be13edd6b10da33"},
    "attention_softmax": {"read": 805359104, "write": 501249792, "src": "2be13edd6b10da33"},
    "chained_ln_gelu_rms": {"read": 115985408, "write": 88527104, "src": "2ebf5273d3cc2d77"},
    "column_layernorm": {"read": 309405696, "write": 99708160, "src": "2ebf5273d3cc2d77"},
    "gelu_rmsnorm": {"read": 118271744, "write": 90887936, "src": "2ebf5273d3cc2d77"},
    "layernorm_256": {"read": 306688, "write": 0, "src": "2ebf5273d3cc2d77"},
    "mlp_b2b": {"read": 50491648, "write": 23822592, "src": "2be13edd6b10da33"},
    "mlp_bottom": {"read": 316160, "write": 0, "rows": 64, "src": "2be13edd6b10da33"},
    "postnorm_layernorm": {"read": 199381504, "write": 92698880, "src": "2ebf5273d3cc2d77"},
    "scaled_softmax": {"read": 1387041024, "write": 239633664, "src": "2ebf5273d3cc2d77"},
    "target_attention": {"read": 15002368, "write": 0, "rows": 64, "src": "2be13edd6b10da33"},
}


# Global store bytes of one fused launch, from the SM-to-L2 store counters
# (`ncu --metrics l1tex__m_l1tex2xbar_write_bytes_mem_global_op_tma_st.sum,
# ..._mem_lg_op_st.sum, ..._mem_global_op_red.sum, ..._mem_global_op_atom.sum`
# on the fused kernel, fp32 output): TMA stores, plain global stores, and the
# 4-byte reductions and atomics on the workspace's arrival counters (counted
# per 32-byte sector).  Keyed and validated like NCU_TRAFFIC.
NCU_STORES = {
    "attention_long_keys": {"tma": 0, "st": 524288, "red": 0, "atom": 0, "src": "2be13edd6b10da33"},
    "attention_relu": {"tma": 0, "st": 536870912, "red": 0, "atom": 0, "src": "2be13edd6b10da33"},
    "attention_softmax": {"tma": 0, "st": 536870912, "red": 0, "atom": 0, "src": "2be13edd6b10da33"},
    "chained_ln_gelu_rms": {"tma": 134217728, "st": 2097152, "red": 262144, "atom": 0, "src": "2ebf5273d3cc2d77"},
    "column_layernorm": {"tma": 134217728, "st": 1048576, "red": 131072, "atom": 0, "src": "2ebf5273d3cc2d77"},
    "gelu_rmsnorm": {"tma": 134217728, "st": 1048576, "red": 131072, "atom": 0, "src": "2ebf5273d3cc2d77"},
    "layernorm_256": {"tma": 262144, "st": 0, "red": 0, "atom": 0, "src": "2ebf5273d3cc2d77"},
    "mlp_b2b": {"tma": 0, "st": 67108864, "red": 0, "atom": 0, "src": "2be13edd6b10da33"},
    "mlp_bottom": {"tma": 0, "st": 65536, "red": 0, "atom": 0, "rows": 64, "src": "2be13edd6b10da33"},
    "postnorm_layernorm": {"tma": 134217728, "st": 1048576, "red": 131072, "atom": 0, "src": "2ebf5273d3cc2d77"},
    "scaled_softmax": {"tma": 268435456, "st": 2097152, "red": 262144, "atom": 0, "src": "2ebf5273d3cc2d77"},
    "target_attention": {"tma": 0, "st": 16777216, "red": 0, "atom": 0, "rows": 64, "src": "2be13edd6b10da33"},
}


class _NotApplicable(Exception):
    """A comparison that the configuration has no counterpart for."""


def percentile(xs, q: float) -> float:
    """Nearest-rank percentile (q in [0, 1]) of a non-empty list."""
    v = sorted(xs)
    return v[min(len(v) - 1, int(round(q * (len(v) - 1))))]


# Cycles of the device-side sleep enqueued ahead of a timed call (about
# 0.1 ms at 2 GHz): the GPU stays busy while the host enqueues the call's
# launches, so the host's launch time never falls inside an event pair.
AHEAD_CYCLES = 200_000


def warm_times(fn, stream, n: int) -> float:
    """Mean CUDA-event time (ms) of `n` back-to-back calls of `fn` on
    `stream`, with nothing between them (no L2 flush), after one untimed
    call.  A bounded device-side sleep (about 0.1 ms per call) is enqueued
    first, so the host has queued every call before the GPU reaches the
    first: no host launch gap falls inside an event pair."""
    fn()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        torch.cuda._sleep(AHEAD_CYCLES * n)
    for k in range(n):
        starts[k].record(stream)
        fn()
        ends[k].record(stream)
    torch.cuda.synchronize()
    return statistics.mean(s.elapsed_time(e) for s, e in zip(starts, ends))


def kernel_source_hash(b2b: bool) -> str:
    """Hash of the sources of the fused kernel family a workload runs."""
    h = hashlib.sha256()
    for f in (("cf_b2b.cu" if b2b else "cf_gemm_epi_kernel.cuh"), "cf_ptx.cuh", "cf_internal.h"):
        with open(os.path.join(ROOT, "back_gemm_fusion_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# ----------------------------------------------------------------- workloads
class Workload:
    """A fused GEMM-epilogue or B2BGEMM problem with its accounting."""

    def __init__(self, name: str, seed: int = 0, exchange: str = "auto", rows: int = 64, out_dtype: str = "fp32"):
        self.name = name
        self.exchange = exchange
        # --rows sizes these two workloads (the bottom MLP's rows, target
        # attention's users); the stored counters hold for one size only.
        self.size_rows = rows if name in ("mlp_bottom", "target_attention") else None
        self.out_dtype = torch.bfloat16 if out_dtype == "bf16" else torch.float32
        ob = 2.0 if out_dtype == "bf16" else 4.0
        if name == "gelu_rmsnorm":
            self.case = I.gelu_rmsnorm(seed)
        elif name == "layernorm_256":
            self.case = I.layernorm_256(seed)
        elif name == "scaled_softmax":
            self.case = I.scaled_softmax(seed)
        elif name == "postnorm_layernorm":
            self.case = I.postnorm_layernorm(seed)
        elif name == "chained_ln_gelu_rms":
            self.case = I.chained_ln_gelu_rms(seed)
        elif name == "column_layernorm":
            self.case = I.column_layernorm(seed)
        elif name == "mlp_b2b":
            self.case = I.mlp_b2b(seed)
        elif name == "mlp_bottom":
            self.case = I.mlp_bottom(seed, rows=rows)
        elif name == "target_attention":
            self.case = I.target_attention(seed, batch=rows)
        elif name == "attention_long_keys":
            self.case = I.attention_long_keys(seed)
        elif name in ("attention_softmax", "attention_relu"):
            op = "scale_softmax" if name == "attention_softmax" else "scale_relu"
            self.case = I.attention_b2b(seed, op=op)
        else:
            raise ValueError(name)
        self.axis = "row"
        self.is_b2b = name in ("mlp_b2b", "mlp_bottom", "attention_softmax", "attention_relu", "target_attention",
                               "attention_long_keys")
        c = self.case
        if not self.is_b2b:
            self.axis = c.meta.get("axis", "row")
        if self.is_b2b:
            self.flops = 2.0 * c.batch * c.M * (c.K * c.N1 + c.N1 * c.N2)
            self.out_bytes = ob * c.batch * c.M * c.N2
            self.bytes = 2.0 * (c.A.numel() + c.W1.numel() + c.W2.numel()) + self.out_bytes
            self.stat_bytes = 0.0
            self.rows = c.batch * c.M
        else:
            vec = sum(t.numel() for t in (c.bias, c.gamma, c.beta, c.stage0_gamma, c.stage0_beta) if t is not None)
            self.flops = 2.0 * c.M * c.N * c.K
            self.out_bytes = ob * c.M * c.N
            res = 0.0 if c.residual is None else float(c.residual.numel() * c.residual.element_size())
            self.bytes = 2.0 * (c.M * c.K + c.K * c.N) + 4.0 * vec + res + self.out_bytes
            # Row statistics of rows wider than one 256-column tile: 8 bytes
            # per row per tile in the workspace (written once, read per tile).
            n_row = sum(o[0] in ("layernorm", "rmsnorm", "softmax") for o in c.ops)
            # Column reductions: per column per 256-row tile.
            lines, length = (c.N, c.M) if self.axis == "col" else (c.M, c.N)
            self.stat_bytes = 8.0 * n_row * lines * (length // 256) if length > 256 else 0.0
            self.rows = c.N if self.axis == "col" else c.M  # oracle sample units

    def config(self):
        c = self.case
        out = "bf16" if self.out_dtype == torch.bfloat16 else "fp32"
        if self.is_b2b:
            return {"workload": self.name, "batch": c.batch, "M": c.M, "K": c.K, "N1": c.N1, "N2": c.N2,
                    "mid_op": c.op, "intermediate": "bf16, on chip", "out": out}
        return {"workload": self.name, "M": c.M, "N": c.N, "K": c.K, "ops": [list(o) for o in c.ops],
                "axis": self.axis, "row_stat_exchange": self.exchange, "out": out}

    # -- GPU side
    def to_device(self):
        c = self.case
        dev = {}
        if self.is_b2b:
            dev["A"], dev["W1"], dev["W2"] = c.A.cuda(), c.W1.cuda(), c.W2.cuda()
            dev["out"] = torch.empty((c.batch, c.M, c.N2), dtype=self.out_dtype, device="cuda")
        else:
            dev["A"] = c.A.cuda()
            # Column reductions take B as its N x K transpose.
            dev["B"] = c.B.t().contiguous().cuda() if self.axis == "col" else c.B.cuda()
            for k in ("bias", "gamma", "beta", "residual", "stage0_gamma", "stage0_beta"):
                t = getattr(c, k)
                dev[k] = None if t is None else t.cuda()
            dev["out"] = torch.empty((c.M, c.N), dtype=self.out_dtype, device="cuda")
        return dev

    def fused_step(self, cf, dev, stream=None, workspace=None):
        c = self.case
        if self.is_b2b:
            A = dev["A"] if c.batch > 1 else dev["A"][0]
            W1 = dev["W1"] if c.batch > 1 else dev["W1"][0]
            W2 = dev["W2"] if c.batch > 1 else dev["W2"][0]
            out = dev["out"] if c.batch > 1 else dev["out"][0]
            cf.cf_b2bgemm(A, W1, W2, c.op, c.scale, w1_trans=c.w1_k_major, out=out, stream=stream)
        else:
            cf.cf_gemm_epilogue(dev["A"], dev["B"], c.ops, dev["bias"], dev["gamma"], dev["beta"],
                                out=dev["out"], workspace=workspace, stream=stream, exchange=self.exchange,
                                residual=dev["residual"], stage0_gamma=dev["stage0_gamma"],
                                stage0_beta=dev["stage0_beta"], b_trans=self.axis == "col", axis=self.axis)

    def unfused_step(self, cf, dev, scratch, stream=None):
        c = self.case
        if self.is_b2b:
            A = dev["A"] if c.batch > 1 else dev["A"][0]
            W1 = dev["W1"] if c.batch > 1 else dev["W1"][0]
            W2 = dev["W2"] if c.batch > 1 else dev["W2"][0]
            out = dev["out"] if c.batch > 1 else dev["out"][0]
            s, p = scratch
            cf.cf_unfused_b2bgemm(A, W1, W2, c.op, c.scale, w1_trans=c.w1_k_major, out=out,
                                  s_buf=s if c.batch > 1 else s[0], p_buf=p if c.batch > 1 else p[0],
                                  stream=stream)
        else:
            cf.cf_unfused_gemm_epilogue(dev["A"], dev["B"], c.ops, dev["bias"], dev["gamma"], dev["beta"],
                                        out=dev["out"], intermediate=scratch, stream=stream,
                                        residual=dev["residual"], stage0_gamma=dev["stage0_gamma"],
                                        stage0_beta=dev["stage0_beta"], b_trans=self.axis == "col", axis=self.axis)

    def unfused_scratch(self):
        c = self.case
        if self.is_b2b:
            return (torch.empty((c.batch, c.M, c.N1), dtype=torch.float32, device="cuda"),
                    torch.empty((c.batch, c.M, c.N1), dtype=torch.bfloat16, device="cuda"))
        return torch.empty((c.M, c.N), dtype=torch.float32, device="cuda")

    # -- oracle side (CPU)
    def _f64(self, key):
        cache = self.__dict__.setdefault("_f64_cache", {})
        if key not in cache:
            cache[key] = I.to_f64(getattr(self.case, key))
        return cache[key]

    def oracle_rows(self, rows):
        """Run the oracle on a subset of output rows (flops of that subset)."""
        from oracle import cf_oracle as O
        c = self.case
        if self.is_b2b:
            # rows index flattened (batch, row) pairs; group by batch entry
            b_idx = rows // c.M
            r_idx = rows % c.M
            for b in np.unique(b_idx):
                rr = r_idx[b_idx == b]
                A = I.to_f64(c.A[b])[rr]
                W1 = I.to_f64(c.W1[b])
                W1 = W1.T if c.w1_k_major else W1
                O.b2bgemm(A, W1, I.to_f64(c.W2[b]), c.op, c.scale)
            return 2.0 * len(rows) * (c.K * c.N1 + c.N1 * c.N2)
        if self.axis == "col":
            # Column reductions: the sampled units are output columns (each
            # needs all M rows).
            def cols(key):
                v = self._f64(key)
                return None if v is None else v[..., rows]
            R = None if c.residual is None else self._f64("residual")[:, rows]
            O.gemm_epilogue(self._f64("A"), self._f64("B")[:, rows], c.ops, cols("bias"), cols("gamma"), cols("beta"),
                            residual=R, stage0_gamma=cols("stage0_gamma"), stage0_beta=cols("stage0_beta"), axis="col")
            return 2.0 * len(rows) * c.M * c.K
        A = self._f64("A")[rows]
        R = None if c.residual is None else self._f64("residual")[rows]
        O.gemm_epilogue(A, self._f64("B"), c.ops, self._f64("bias"), self._f64("gamma"), self._f64("beta"),
                        residual=R, stage0_gamma=self._f64("stage0_gamma"), stage0_beta=self._f64("stage0_beta"))
        return 2.0 * len(rows) * c.N * c.K


# ----------------------------------------------------------------- helpers
class NvmlSampler:
    """Samples SM clocks and clock-event (throttle) reasons through NVML
    (libnvidia-ml via ctypes, read-only queries) every ~1 ms while running."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, torch_index: int):
        import ctypes
        import threading
        self.ok = False
        self.samples = []
        self.reasons = 0
        self.stop = threading.Event()
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                return
            props = torch.cuda.get_device_properties(torch_index)
            bus = "%08x:%02x:%02x.0" % (getattr(props, "pci_domain_id", 0), props.pci_bus_id, props.pci_device_id)
            h = ctypes.c_void_p()
            if lib.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(h)) != 0:
                return
            mx = ctypes.c_uint()
            lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx))
            self.max_mhz = mx.value
            self.lib, self.h, self.ctypes = lib, h, ctypes
            self.reason_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons")
            self.ok = True
        except Exception:
            self.ok = False

    def _run(self):
        c = self.ctypes
        clk, rs = c.c_uint(), c.c_ulonglong()
        while not self.stop.is_set():
            if self.lib.nvmlDeviceGetClockInfo(self.h, 1, c.byref(clk)) == 0:
                self.samples.append(clk.value)
            if self.reason_fn(self.h, c.byref(rs)) == 0:
                self.reasons |= rs.value
            time.sleep(0.001)

    def __enter__(self):
        import threading
        if self.ok:
            self.t = threading.Thread(target=self._run, daemon=True)
            self.t.start()
        return self

    def __exit__(self, *exc):
        if self.ok:
            self.stop.set()
            self.t.join()

    def summary(self):
        if not self.ok or not self.samples:
            return None
        return {"sm_mhz": statistics.median(self.samples), "sm_max_mhz": self.max_mhz,
                "reasons": [n for b, n in self.REASONS.items() if self.reasons & b],
                "samples": len(self.samples), "source": "nvml"}


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while running."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.idx = device_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if self.proc is None or not self.path:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sms, maxes, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sms.append(float(parts[1]))
                    maxes.append(float(parts[2]))
                except ValueError:
                    continue
                for nm, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(nm)
        os.unlink(self.path)
        if not sms:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        load = [s for s in sms if s > 0.5 * max(sms)] or sms
        return {"sm_mhz": statistics.median(load), "sm_max_mhz": max(maxes), "reasons": sorted(reasons),
                "samples": len(sms)}


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
        return dist, rank, world, local
    return None, 0, 1, 0


def barrier(dist):
    if dist is not None:
        dist.barrier()


def max_over_ranks(dist, v: float) -> float:
    if dist is None:
        return v
    t = torch.tensor([v], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def time_oracle(wl: Workload, budget_s: float, resize: bool = True):
    """Time the oracle on a seeded row sample sized to about budget_s seconds
    (resize: size it once more when the first sample ran well under budget;
    the reference arm's many short steps skip that)."""
    rng = np.random.default_rng(0)
    n = 16 if wl.is_b2b else 64
    t0 = time.perf_counter()
    flops = wl.oracle_rows(np.sort(rng.choice(wl.rows, size=min(n, wl.rows), replace=False)))
    dt = time.perf_counter() - t0
    rows = int(min(wl.rows, max(n, n * budget_s / max(dt, 1e-3))))
    for _ in range(2 if resize else 1):
        sample = np.sort(rng.choice(wl.rows, size=rows, replace=False))
        t0 = time.perf_counter()
        flops = wl.oracle_rows(sample)
        dt = time.perf_counter() - t0
        # The small pilot over-estimates the cost per row (fixed costs per
        # call): size the sample once more when it ran well under budget.
        if dt >= 0.6 * budget_s or rows >= wl.rows:
            break
        rows = int(min(wl.rows, rows * budget_s / max(dt, 1e-3)))
    return flops / dt / 1e12, rows, dt


# ----------------------------------------------------------------- arms
def run_reference(args, wl: Workload, dist, rank, world):
    if rank != 0:
        return
    cores = os.cpu_count()
    for _ in range(args.warmup):
        time_oracle(wl, args.ref_step_seconds / 4, resize=False)
    vals, rows_used, secs = [], 0, 0.0
    for _ in range(args.steps):
        v, rows_used, dt = time_oracle(wl, args.ref_step_seconds, resize=False)
        vals.append(v)
        secs += dt
    value = statistics.mean(vals)
    unit = "columns" if getattr(wl, "axis", "row") == "col" else "rows"
    sample = f"{rows_used} of {wl.rows} output {unit} (seeded), float64 numpy oracle, extrapolated per {unit[:-1]}"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * secs / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": wl.config(),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def measure(args, wl: Workload, cf, peaks, dist, rank, world, local, steps: int, warmup: int,
            cpu_seconds: float, variants: bool = True):
    """Time one workload: the fused call (CUDA events over `steps` steps, L2
    flushed between them), the unfused path and the other exchanges in the
    same run, the end-to-end call with host buffers, and the oracle on a
    bounded host sample.  Returns the per-workload record (rank 0)."""
    dev = wl.to_device()
    stream = torch.cuda.current_stream()
    workspace = None
    if not wl.is_b2b:
        c = wl.case
        need = cf.cf_workspace_size(dev["A"], dev["B"], c.ops, exchange=wl.exchange, b_trans=wl.axis == "col",
                                    axis=wl.axis)
        if need:
            workspace = torch.empty(need, dtype=torch.uint8, device="cuda")
    flush = torch.empty(256 * 2 ** 20 // 4, dtype=torch.float32, device="cuda")

    def step():
        wl.fused_step(cf, dev, stream, workspace)

    for _ in range(warmup):
        flush.fill_(1.0)
        step()
    torch.cuda.synchronize()
    if cf.cf_last_device_status() != 0:
        raise RuntimeError(f"{wl.name}: device status reports a timeout after warm-up")
    # Other row-statistics exchanges of the same fused kernel, same run.
    xvar = {}
    if variants and not wl.is_b2b and any(o[0] in ("layernorm", "rmsnorm", "softmax") for o in wl.case.ops):
        for xch in ("cluster", "global", "global_dynamic"):
            if xch == wl.exchange:
                continue
            try:
                wv = Workload.__new__(Workload)
                wv.__dict__.update(wl.__dict__)
                wv.exchange = xch
                ws = workspace
                if ws is None:
                    need = cf.cf_workspace_size(dev["A"], dev["B"], wl.case.ops, exchange=xch,
                                                b_trans=wl.axis == "col", axis=wl.axis)
                    ws = torch.empty(need, dtype=torch.uint8, device="cuda") if need else None
                for _ in range(2):
                    wv.fused_step(cf, dev, stream, ws)
                torch.cuda.synchronize()
                vm = []
                for k in range(max(3, steps)):
                    torch.cuda._sleep(AHEAD_CYCLES)
                    flush.fill_(float(k))
                    s0, e0 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    s0.record(stream)
                    wv.fused_step(cf, dev, stream, ws)
                    e0.record(stream)
                    torch.cuda.synchronize()
                    vm.append(s0.elapsed_time(e0))
                v = statistics.mean(vm)
                xvar[xch] = {"ms_per_step": v, "tflops": wl.flops / (v * 1e-3) / 1e12}
            except Exception as exc:
                xvar[xch] = {"error": str(exc)[:200]}

    # Unfused comparison (cuBLASLt GEMM + separate epilogue kernel), same run.
    unfused = None
    bf16_out = str(dev["out"].dtype) == "torch.bfloat16"
    try:
        if bf16_out and not wl.is_b2b:
            raise _NotApplicable("the unfused GEMM-epilogue comparison path writes fp32 output only")
        scratch = wl.unfused_scratch()
        for _ in range(2):
            wl.unfused_step(cf, dev, scratch, stream)
        torch.cuda.synchronize()
        um = []
        for k in range(max(3, steps)):
            torch.cuda._sleep(AHEAD_CYCLES)  # the unfused path is several direct launches
            flush.fill_(float(k))
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record(stream)
            wl.unfused_step(cf, dev, scratch, stream)
            e.record(stream)
            torch.cuda.synchronize()
            um.append(s.elapsed_time(e))
        u = statistics.mean(um)
        uw = warm_times(lambda: wl.unfused_step(cf, dev, scratch, stream), stream, max(3, steps))
        unfused = {"ms_per_step": u, "tflops": wl.flops / (u * 1e-3) / 1e12, "warm_l2_ms_per_step": uw,
                   "path": ("cuBLASLt GEMM1 -> HBM S -> mid-op kernel -> HBM bf16 S' -> cuBLASLt GEMM2"
                            if wl.is_b2b else "cuBLASLt GEMM -> HBM intermediate -> separate epilogue kernel")}
        del scratch
    except _NotApplicable as exc:
        unfused = {"unavailable": str(exc)}
    except Exception as exc:  # the comparison path is optional for the headline
        unfused = {"error": str(exc)[:200]}

    # The fused call captured once in a CUDA graph and replayed: the device
    # time of a small problem is then not the host's marshalling and launch
    # time (the graph holds the same launch, with the same arguments).
    graph, launch_mode = None, "direct"
    if not args.no_graph:
        try:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                wl.fused_step(cf, dev, None, workspace)
            g.replay()
            torch.cuda.synchronize()
            if cf.cf_last_device_status() != 0:
                raise RuntimeError("device status reports a timeout in the graph replay")
            graph, launch_mode = g, "cuda graph replay"
        except Exception as exc:  # direct launches remain valid; say why
            launch_mode = f"direct (graph capture failed: {str(exc)[:120]})"
            torch.cuda.synchronize()

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    with ClockSampler(local) as clk, NvmlSampler(torch.cuda.current_device()) as nv:
        barrier(dist)
        torch.cuda.synchronize()
        t_wall = time.perf_counter()
        for k in range(steps):
            flush.fill_(float(k))
            starts[k].record(stream)
            if graph is not None:
                graph.replay()
            else:
                step()
            ends[k].record(stream)
        torch.cuda.synchronize()
        barrier(dist)
        t_wall = time.perf_counter() - t_wall
    clocks = nv.summary() or clk.summary()
    if cf.cf_last_device_status() != 0:
        raise RuntimeError(f"{wl.name}: device status reports a timeout in the timed region")
    ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    ms_step = max_over_ranks(dist, statistics.mean(ms))
    tflops = wl.flops / (ms_step * 1e-3) / 1e12
    value = tflops * world
    if unfused and "ms_per_step" in unfused:
        unfused["fused_speedup"] = unfused["ms_per_step"] / ms_step
    # Warm L2: the same launch back to back with no flush in between, so
    # that inputs no larger than L2 stay cached (the small configurations'
    # usual case inside a model).  Reported beside the flushed figure.
    warm_ms = warm_times(graph.replay if graph is not None else step, stream, max(3, steps))
    if cf.cf_last_device_status() != 0:
        raise RuntimeError(f"{wl.name}: device status reports a timeout in the warm-L2 steps")
    warm = {"ms_per_step": warm_ms, "tflops": wl.flops / (warm_ms * 1e-3) / 1e12, "launch": launch_mode}
    if unfused and "warm_l2_ms_per_step" in unfused:
        warm["unfused_ms_per_step"] = unfused["warm_l2_ms_per_step"]
        warm["fused_speedup"] = unfused["warm_l2_ms_per_step"] / warm_ms
    del graph

    # End to end through the public API: pinned host inputs -> device, fused
    # call, device -> pinned host output, all inside the timed region.
    c = wl.case
    host_in = []
    names = ("A", "W1", "W2") if wl.is_b2b else ("A", "B", "bias", "gamma", "beta", "residual", "stage0_gamma",
                                                  "stage0_beta")
    for k in names:
        t = getattr(c, k)
        if t is not None:
            if k == "B" and wl.axis == "col":
                t = t.t().contiguous()  # the device copy is B's N x K transpose
            host_in.append((k, t.pin_memory()))
    host_out = torch.empty(dev["out"].shape, dtype=dev["out"].dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for _, t in host_in)
    d2h = host_out.numel() * host_out.element_size()
    e2e_ms = []
    for k in range(max(3, steps)):
        torch.cuda.synchronize()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        for name, t in host_in:
            dev[name].copy_(t, non_blocking=True)
        step()
        host_out.copy_(dev["out"], non_blocking=True)
        e.record(stream)
        torch.cuda.synchronize()
        e2e_ms.append(s.elapsed_time(e))
    e2e_step = max_over_ranks(dist, statistics.mean(e2e_ms))
    e2e_val = wl.flops / (e2e_step * 1e-3) / 1e12 * world
    if cf.cf_last_device_status() != 0:
        raise RuntimeError(f"{wl.name}: device status reports a timeout in the end-to-end steps")
    del dev, workspace, flush, host_in, host_out
    torch.cuda.synchronize()
    torch.cuda.empty_cache()

    if rank != 0:
        return None
    # CPU baseline: the oracle on the host cores, bounded sample.
    ref_tflops, ref_rows, ref_s = time_oracle(wl, cpu_seconds)
    t_roof = max(wl.flops / (peaks["bf16_tflops"] * 1e12), wl.bytes / (peaks["hbm_gbs"] * 1e9))
    src = kernel_source_hash(wl.is_b2b)
    fp32 = wl.out_dtype == torch.float32  # counters taken with fp32 out
    def counters_hold(entry):
        return entry and entry.get("src") == src and entry.get("rows") == wl.size_rows

    tr = NCU_TRAFFIC.get(wl.name) if fp32 else None
    tr = tr if counters_hold(tr) else None
    traffic = (tr["read"] + tr["write"]) if tr else None
    # The page's own test: global store bytes of one launch beyond the
    # output and the row-statistics workspace (an intermediate would have
    # to be stored), from the store counters; the counter updates are
    # listed apart.
    stc = NCU_STORES.get(wl.name) if fp32 else None
    stc = stc if counters_hold(stc) else None
    inter = (stc["tma"] + stc["st"] - wl.out_bytes - wl.stat_bytes) if stc else None
    return {
        "workload": wl.name, "value": value, "ms_per_step": ms_step, "tflops": tflops,
        "ms_per_step_dist": {"p10": percentile(ms, 0.1), "median": statistics.median(ms), "p90": percentile(ms, 0.9),
                             "mean": statistics.mean(ms), "rank": rank},
        "config": {**wl.config(), "l2": "flushed between timed steps (256 MB write)", "launch": launch_mode,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "roofline": {"bound": "tensor", "achieved": tflops, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": tflops / peaks["bf16_tflops"], "traffic": traffic,
                     "peak_source": f"{peaks['source']} bf16 burst",
                     "roofline_frac": (t_roof * 1e3) / ms_step},
        "warm_l2": warm,
        "intermediate_hbm_bytes": inter,
        "global_store_bytes": ({"tma_stores": stc["tma"], "stores": stc["st"], "counter_updates": stc["red"] + stc["atom"],
                                "output": wl.out_bytes, "row_stats": wl.stat_bytes,
                                "source": "ncu SM-to-L2 store counters, one launch"} if stc else None),
        "dram_bytes": ({"read": tr["read"], "write": tr["write"], "source": "ncu, one launch"} if tr else None),
        "compulsory_bytes": wl.bytes,
        "cpu_baseline": {"value": ref_tflops, "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
                         "sample": f"{ref_rows} of {wl.rows} output {'columns' if wl.axis == 'col' else 'rows'} "
                                   f"(seeded), {ref_s:.1f} s"},
        "e2e": {"value": e2e_val, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_step},
        "unfused": unfused,
        "exchange_variants": xvar or None,
        "gpu_launches": steps,
        "clocks": clocks,
        "wall_s_timed_region": t_wall,
        "kernel_src": src,
    }


# The configurations the metric is quoted on, by workload name: the GEMM +
# bias + LayerNorm latency case, GELU + RMSNorm, the softmax logit head, the
# MLP B2BGEMM and both attention variants.
CONFIG_WORKLOADS = ["layernorm_256", "gelu_rmsnorm", "scaled_softmax", "mlp_b2b", "attention_softmax",
                    "attention_relu"]


def run_ours(args, wl: Workload, dist, rank, world, local):
    import back_gemm_fusion_gb300 as cf
    from back_gemm_fusion_gb300 import build
    build.build()
    cf.load_library()
    peaks = load_peaks()
    if args.once:
        # One fused launch and nothing else (for a profiler's kernel filter).
        dev = wl.to_device()
        workspace = None
        if not wl.is_b2b:
            need = cf.cf_workspace_size(dev["A"], dev["B"], wl.case.ops, exchange=wl.exchange,
                                        b_trans=wl.axis == "col", axis=wl.axis)
            workspace = torch.empty(need, dtype=torch.uint8, device="cuda") if need else None
        wl.fused_step(cf, dev, torch.cuda.current_stream(), workspace)
        torch.cuda.synchronize()
        st = cf.cf_last_device_status()
        print(json.dumps({"workload": wl.name, "once": True, "device_status": st}), flush=True)
        if st != 0:
            raise RuntimeError("device status reports a timeout")
        return
    head = measure(args, wl, cf, peaks, dist, rank, world, local, args.steps, args.warmup, args.cpu_seconds)
    configs = {}
    if args.configs == "all":
        for name in CONFIG_WORKLOADS:
            if name == wl.name and wl.out_dtype == torch.float32 and wl.exchange == "auto":
                continue
            w2 = Workload(name, exchange="auto", rows=args.rows)
            r = measure(args, w2, cf, peaks, dist, rank, world, local, args.config_steps, 3, args.config_cpu_seconds,
                        variants=False)
            del w2
            if r is not None:
                configs[name] = {k: r[k] for k in ("value", "ms_per_step", "ms_per_step_dist", "config", "roofline",
                                                   "intermediate_hbm_bytes", "global_store_bytes", "dram_bytes",
                                                   "compulsory_bytes", "cpu_baseline", "e2e", "unfused",
                                                   "warm_l2", "gpu_launches", "clocks")}
                configs[name]["steps"] = args.config_steps
    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": head["value"], "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "ms_per_step_dist": head["ms_per_step_dist"],
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": head["config"],
        "roofline": head["roofline"],
        "intermediate_hbm_bytes": head["intermediate_hbm_bytes"],
        "global_store_bytes": head["global_store_bytes"],
        "dram_bytes": head["dram_bytes"],
        "compulsory_bytes": head["compulsory_bytes"],
        "cpu_baseline": head["cpu_baseline"],
        "e2e": head["e2e"],
        "unfused": head["unfused"],
        "warm_l2": head["warm_l2"],
        "exchange_variants": head["exchange_variants"],
        "gpu_launches": head["gpu_launches"],
        "clocks": head["clocks"],
        "wall_s_timed_region": head["wall_s_timed_region"],
        "kernel_src": head["kernel_src"],
        "configs": configs or None,
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="attention_softmax",
                    choices=["gelu_rmsnorm", "layernorm_256", "scaled_softmax", "mlp_b2b", "attention_softmax",
                             "attention_relu", "mlp_bottom", "postnorm_layernorm", "chained_ln_gelu_rms",
                             "target_attention", "column_layernorm", "attention_long_keys"])
    ap.add_argument("--rows", type=int, default=64,
                    help="batch of the mlp_bottom (rows) and target_attention (users) workloads (1..64)")
    ap.add_argument("--exchange", default="auto", choices=["auto", "cluster", "global", "global_dynamic"],
                    help="row-statistics exchange of the fused GEMM-epilogue kernel")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="budget of the CPU-baseline oracle sample")
    ap.add_argument("--ref-step-seconds", type=float, default=5.0, help="oracle seconds per reference step")
    ap.add_argument("--out-dtype", default="fp32", choices=["fp32", "bf16"],
                    help="output dtype of the fused call (the unfused GEMM-epilogue path is fp32-only)")
    ap.add_argument("--no-graph", action="store_true",
                    help="time direct launches instead of replaying the fused call's CUDA graph")
    ap.add_argument("--configs", default="all", choices=["all", "none"],
                    help="also measure every other configuration of the metric (the 'configs' object)")
    ap.add_argument("--config-steps", type=int, default=10, help="timed steps per extra configuration")
    ap.add_argument("--config-cpu-seconds", type=float, default=4.0,
                    help="oracle sample budget per extra configuration")
    ap.add_argument("--once", action="store_true",
                    help="run the fused kernel of the workload once and exit (profiling captures)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3) if args.impl == "ours" else args.warmup
    dist, rank, world, local = dist_setup(args)
    wl = Workload(args.workload, exchange=args.exchange, rows=args.rows, out_dtype=args.out_dtype)
    if args.impl == "reference":
        run_reference(args, wl, dist, rank, world)
    else:
        run_ours(args, wl, dist, rank, world, local)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
