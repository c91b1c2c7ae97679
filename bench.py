"""Benchmark of the packed double-binary matmul on B300.

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--no-also]

One step = one pass of the hot path over one batch of synthetic input: for the
decode workloads, L back-to-back dbf_matmul calls, each on its own factor set,
activations and outputs (L chosen so one step touches more than 4x the L2
cache, so no timed step is served from L2), captured in one CUDA graph with
programmatic dependent launch between the kernels.  The headline workload is
the LoRDBA adapter branch on a 4096x4096 projection (R=64, ell=1) at T=16
decode tokens.  `value` is tokens per second through one projection call,
summed over all ranks; `roofline` compares the per-call algorithmic bytes
(sign bits + fp16 scales + x + y) per call duration with the measured HBM
copy bandwidth.  The other workloads (1.5-bit DBF projection, the DBF MLP in
prefill, multi-adapter serving, the tiny case) are measured the same way and
reported under "also".

--impl reference times the fp64 CPU oracle on the host cores instead (the
same metric on a bounded sample of the headline workload).
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from workloads import configs as CFG  # noqa: E402
from workloads import generators as G  # noqa: E402

METRIC = "tokens/s + % roofline: HBM GB/s (decode T≤16), tensor-pipe util (T=2048)"
L2_BYTES = 126 * 1024 * 1024
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}


# --------------------------------------------------------------------- setup

def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-also", action="store_true", help="skip the secondary workloads")
    ap.add_argument("--only", default=None, help="run only this secondary workload key")
    ap.add_argument("--workload", default="adapter4k_T16",
                    help="workload timed for the main line (default: the headline adapter4k_T16)")
    ap.add_argument("--max-calls", type=int, default=None,
                    help="cap on calls per step (small profiling runs; breaks the > 4x L2 rule)")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-io end-to-end leg")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline leg")
    ap.add_argument("--no-single", action="store_true", help="skip the cold-L2 single-call latency leg")
    return ap.parse_args(argv)


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            d = json.load(fh)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def sources_hash(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "double_binary_rank_packed_b300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_traffic(workload_key):
    """DRAM bytes per launch of the workload's dominant kernel, from the committed ncu
    summary (profiles/dram_traffic.json), or None when the kernel sources changed since."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as fh:
        d = json.load(fh)
    e = d.get(workload_key)
    if not e or sources_hash(e["sources"]) != e.get("sources_hash"):
        return None
    return e.get("dram_bytes_per_launch")


def aggregate(local_ms: float, local_units: float, dist_mod=None):
    """Max elapsed time over ranks and the sum of units: (max_ms, total_units)."""
    if dist_mod is None:
        return local_ms, local_units
    import torch
    t = torch.tensor([local_ms], dtype=torch.float64)
    u = torch.tensor([local_units], dtype=torch.float64)
    if dist_mod.get_backend() == "nccl":
        t, u = t.cuda(), u.cuda()
    dist_mod.all_reduce(t, op=dist_mod.ReduceOp.MAX)
    dist_mod.all_reduce(u, op=dist_mod.ReduceOp.SUM)
    return float(t.item()), float(u.item())


# ------------------------------------------------------------- clock sampling

class _Nvml:
    """Minimal NVML access through ctypes (libnvidia-ml ships with the driver)."""

    NVML_CLOCK_SM = 1

    def __init__(self, index):
        import ctypes
        self.ct = ctypes
        lib = None
        for name in ("libnvidia-ml.so.1", "libnvidia-ml.so"):
            try:
                lib = ctypes.CDLL(name)
                break
            except OSError:
                continue
        if lib is None:
            raise OSError("libnvidia-ml not found")
        self.lib = lib
        if lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.h = ctypes.c_void_p()
        if lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index), ctypes.byref(self.h)) != 0:
            raise OSError("nvmlDeviceGetHandleByIndex failed")
        fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None)
        self.reasons_fn = fn if fn is not None else lib.nvmlDeviceGetCurrentClocksThrottleReasons

    def _clock(self, fn):
        v = self.ct.c_uint()
        if fn(self.h, self.ct.c_int(self.NVML_CLOCK_SM), self.ct.byref(v)) != 0:
            raise OSError("clock query failed")
        return int(v.value)

    def sm_mhz(self):
        return self._clock(self.lib.nvmlDeviceGetClockInfo)

    def max_sm_mhz(self):
        return self._clock(self.lib.nvmlDeviceGetMaxClockInfo)

    def reasons(self):
        v = self.ct.c_ulonglong()
        if self.reasons_fn(self.h, self.ct.byref(v)) != 0:
            raise OSError("reasons query failed")
        return int(v.value)


class ClockSampler:
    """Samples SM clock and throttle reasons through NVML while running."""

    REASONS = {
        "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20, "hw_thermal_slowdown": 0x40,
        "hw_power_brake_slowdown": 0x80, "sw_power_cap": 0x4,
    }

    def __init__(self, device_index: int, period_s: float = 0.005):
        self.samples = []
        self.reasons = set()
        self.ok = False
        self.max_mhz = None
        self.period = period_s
        try:
            self.nv = _Nvml(device_index)
            self.max_mhz = self.nv.max_sm_mhz()
            self.ok = True
        except Exception as e:  # no NVML: clocks reported as unavailable
            self.err = repr(e)
            self.ok = False
        self._stop = threading.Event()
        self._t = None

    def _run(self):
        while not self._stop.is_set():
            try:
                self.samples.append(self.nv.sm_mhz())
                mask = self.nv.reasons()
                for name, bit in self.REASONS.items():
                    if mask & bit:
                        self.reasons.add(name)
            except Exception:
                pass
            time.sleep(self.period)

    def __enter__(self):
        if self.ok:
            self._t = threading.Thread(target=self._run, daemon=True)
            self._t.start()
        return self

    def __exit__(self, *exc):
        if self._t is not None:
            self._stop.set()
            self._t.join()

    def summary(self):
        if not self.ok or not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": ["unavailable"], "samples": 0}
        return {"sm_mhz": float(statistics.median(self.samples)), "sm_max_mhz": self.max_mhz,
                "reasons": sorted(self.reasons), "samples": len(self.samples)}


# ------------------------------------------------------------ device inputs

def to_device_factors(dbf, f):
    import torch
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    return dbf.PackedFactors.from_signs(t(f.B1), t(f.B2), t(f.alpha), t(f.beta), t(f.gamma))


def clone_factors(dbf, pf):
    """A copy of a factor set in fresh device memory (a transposed set clones into the plain
    descriptor of the same product)."""
    return dbf.PackedFactors(pf.B1w.clone(), pf.B2w.clone(), pf.alpha.clone(), pf.beta.clone(),
                             pf.gamma.clone(), pf.N, pf.M, pf.R)


def bf16_dev(bits):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def call_footprint(N, M, R, ell, T, ldw1, ldw2):
    return N * ldw1 * 4 + R * ldw2 * 4 + 2 * ell * (N + R + M) + 2 * T * (M + N)


# ---------------------------------------------------------------- workloads

class DecodeWorkload:
    """L independent dbf_matmul calls per step (streamed decode)."""

    def __init__(self, dbf, key, proj, T, outlier_scale=0.0, max_calls=4096, transposed=False, one_launch=False):
        """transposed: time the backward product dx = dy dW (dy [T, N] -> dx [T, M]) through the
        transposed factors instead of the forward one.  one_launch: the two decode stages in one
        cooperative launch with a grid-wide barrier (dbf_selftest_decode_one_launch), the
        comparison arm of the two launches dbf_matmul makes for large R."""
        import torch
        self.dbf, self.key, self.T = dbf, key, T
        self.N, self.M, self.R, self.ell = proj.N, proj.M, proj.R, proj.ell
        f = G.make_factors(proj.N, proj.M, proj.R, proj.ell, proj.seed, proj.sign_mode, proj.scale_mode)
        base = to_device_factors(dbf, f)
        fp = call_footprint(self.N, self.M, self.R, self.ell, T, base.B1w.shape[1], base.B2w.shape[1])
        self.L = int(min(max_calls, max(8, math.ceil(4 * L2_BYTES / fp))))
        if transposed:
            base = dbf.TransposedFactors(base)
            xb = G.make_x(T, proj.N, proj.seed + 7)
        else:
            xb = G.make_x(T, proj.M, proj.seed, outlier_scale=outlier_scale)
        x0 = bf16_dev(xb)
        self.factors = [base] + [clone_factors(dbf, base) for _ in range(self.L - 1)]
        self.x = [x0] + [x0.clone() for _ in range(self.L - 1)]
        self.y = [torch.empty((T, base.N), dtype=torch.bfloat16, device="cuda") for _ in range(self.L)]
        self.ws = dbf.new_workspace(dbf.workspace_bytes(base, T), "cuda")
        self.launches_per_call = dbf.launch_count(base, T)
        self.one_launch = one_launch
        if one_launch:
            self.ws = dbf.new_workspace(dbf.workspace_bytes(base, T, dbf.PATH_DECODE), "cuda")
            self.barrier = torch.zeros(2, dtype=torch.int32, device="cuda")
            self.launches_per_call = 1
        self.fp_call = fp
        self.bytes_per_call = CFG.algorithmic_bytes(self.N, self.M, self.R, self.ell, T)
        self.flops_per_call = CFG.flops(self.N, self.M, self.R, self.ell, T)
        self.bound = "hbm"
        self.graph = None

    def run_eager(self):
        for l in range(self.L):
            self.call_one(l)

    def call_one(self, l):
        if self.one_launch:
            self.dbf.selftest_decode_one_launch(self.factors[l], self.x[l], self.barrier, self.y[l],
                                                workspace=self.ws)
        else:
            self.dbf.matmul(self.factors[l], self.x[l], self.y[l], workspace=self.ws)

    def footprint_per_step(self):
        return self.L * self.fp_call

    def capture(self):
        import torch
        self.run_eager()
        torch.cuda.synchronize()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            self.run_eager()
        torch.cuda.synchronize()
        self.graph = g

    def step(self):
        self.graph.replay()

    @property
    def calls(self):
        return self.L

    @property
    def tokens_per_step(self):
        return self.L * self.T


class PrefillWorkload:
    """The DBF MLP layer: up- and down-projection calls per step (or, transposed, their
    backward products dx = dy dW)."""

    def __init__(self, dbf, key, projs, T, transposed=False):
        import torch
        self.dbf, self.key, self.T = dbf, key, T
        self.items = []
        for p in projs:
            f = G.make_factors(p.N, p.M, p.R, p.ell, p.seed, p.sign_mode, p.scale_mode)
            pf = to_device_factors(dbf, f)
            if transposed:
                pf = dbf.TransposedFactors(pf)
                x = bf16_dev(G.make_x(T, p.N, p.seed + 7))
            else:
                x = bf16_dev(G.make_x(T, p.M, p.seed))
            y = torch.empty((T, pf.N), dtype=torch.bfloat16, device="cuda")
            ws = dbf.new_workspace(dbf.workspace_bytes(pf, T), "cuda")
            self.items.append((pf, x, y, ws, p))
            del f
        self.L = len(self.items)
        self.launches_per_call = dbf.launch_count(self.items[0][0], T)
        self.bytes_per_call = sum(CFG.algorithmic_bytes(p.N, p.M, p.R, p.ell, T) for *_, p in self.items) / self.L
        self.flops_per_call = sum(CFG.flops(p.N, p.M, p.R, p.ell, T) for *_, p in self.items) / self.L
        self.bound = "tensor"
        self.graph = None

    def run_eager(self):
        for pf, x, y, ws, _ in self.items:
            self.dbf.matmul(pf, x, y, workspace=ws)

    capture = DecodeWorkload.capture
    step = DecodeWorkload.step

    def footprint_per_step(self):
        return sum(call_footprint(p.N, p.M, p.R, p.ell, self.T, pf.B1w.shape[1], pf.B2w.shape[1])
                   for pf, _, _, _, p in self.items)

    @property
    def calls(self):
        return self.L

    @property
    def tokens_per_step(self):
        return self.L * self.T


class BackwardWorkload:
    """The backward pass of the DBF MLP layer: one dbf_backward call (dx and the scale gradients
    dalpha, dbeta, dgamma) per projection per step."""

    def __init__(self, dbf, key, projs, T):
        import torch
        self.dbf, self.key, self.T = dbf, key, T
        self.items = []
        for p in projs:
            f = G.make_factors(p.N, p.M, p.R, p.ell, p.seed, p.sign_mode, p.scale_mode)
            pf = to_device_factors(dbf, f)
            ft = dbf.TransposedFactors(pf)
            x = bf16_dev(G.make_x(T, p.M, p.seed))
            dy = bf16_dev(G.make_x(T, p.N, p.seed + 7))
            out = (torch.empty((T, p.M), dtype=torch.bfloat16, device="cuda"),
                   torch.empty((p.ell, p.N), dtype=torch.float32, device="cuda"),
                   torch.empty((p.ell, p.R), dtype=torch.float32, device="cuda"),
                   torch.empty((p.ell, p.M), dtype=torch.float32, device="cuda"))
            ws = dbf.new_workspace(dbf.backward_workspace_bytes(pf, T), "cuda")
            self.items.append((pf, ft, x, dy, out, ws, p))
            del f
        self.L = len(self.items)
        self.launches_per_call = 6  # two prologues and four GEMMs (dbf_backward)
        # x, dy read; dx written; signs read in both orientations; scales read; gradients written
        self.bytes_per_call = sum(2 * T * (p.M + p.N) + 2 * T * p.M + 2 * (p.R * (p.N + p.M)) // 8
                                  + 2 * p.ell * (p.N + p.R + p.M) + 4 * p.ell * (p.N + p.R + p.M)
                                  for *_, p in self.items) / self.L
        # four GEMMs: the forward recomputed (x -> V -> dalpha) and the transposed product (dy -> V' -> dx)
        self.flops_per_call = sum(2 * CFG.flops(p.N, p.M, p.R, p.ell, T) for *_, p in self.items) / self.L
        self.bound = "tensor"
        self.graph = None

    def run_eager(self):
        for pf, ft, x, dy, out, ws, _ in self.items:
            self.dbf.backward(pf, ft, x, dy, workspace=ws, out=out)

    capture = DecodeWorkload.capture
    step = DecodeWorkload.step

    def footprint_per_step(self):
        return sum(2 * call_footprint(p.N, p.M, p.R, p.ell, self.T, pf.B1w.shape[1], pf.B2w.shape[1])
                   for pf, _, _, _, _, _, p in self.items)

    @property
    def calls(self):
        return self.L

    @property
    def tokens_per_step(self):
        return self.L * self.T


# The 1.5 bits/weight layer of the DBF page (k(N+M)/(NM) = 1.5 at N = M = 4096).
FACT_SHAPE = (4096, 4096, 3072)
FACT_SCHED = {"inner": 10, "power_iters": 8, "rho_rel": 1.0}
FP32_LANES_PER_SM = 128
MAX_SM_MHZ = 2032


def factorize_step_flops(n, p, k, inner):
    """Algorithmic FLOPs of one ADMM step fitting an [n x k] factor to T [n x p]: F F^T, T F^T,
    the inverse of F F^T + rho I (k^3: Cholesky, triangular inverse, product), and per
    iteration the P-update (RHS times the inverse)."""
    return 2 * k * k * p + 2 * n * k * p + k ** 3 + inner * 2 * n * k * k


class FactorizeWorkload:
    """One alternating round (A-step, then B-step) of the double binary factorization of a dense
    4096 x 4096 weight at k = 3072: 10 ADMM iterations per step, 8 power iterations per SVID.
    Run eagerly (about 1100 launches per round, each longer than its launch)."""

    def __init__(self, dbf, key):
        import numpy as np
        import torch
        N, M, k = FACT_SHAPE
        self.dbf, self.key, self.N, self.M, self.k = dbf, key, N, M, k
        self.W = torch.from_numpy(G.make_dense_weight(N, M, 4096)).cuda()
        self.f = [torch.from_numpy(np.ascontiguousarray(a)).cuda() for a in G.make_factorize_start(N, M, k, 4096)]
        self.ws = dbf.new_workspace(dbf.factorize_workspace_bytes(N, M, k), "cuda")
        self.calls = 1
        self.T = 0
        self.tokens_per_step = 0
        self.launches_per_call = dbf.factorize_launch_count(N, M, k, 1, **FACT_SCHED)
        inner = FACT_SCHED["inner"]
        self.flops_per_call = factorize_step_flops(N, M, k, inner) + factorize_step_flops(M, N, k, inner)
        self.bytes_per_call = 0
        self.bound = "alu"
        sms = torch.cuda.get_device_properties(0).multi_processor_count
        self.alu_peak_tflops = sms * FP32_LANES_PER_SM * 2 * MAX_SM_MHZ * 1e6 / 1e12
        self.alu_peak_source = (f"derived: {sms} SMs x {FP32_LANES_PER_SM} fp32 lanes x 2 x {MAX_SM_MHZ} MHz "
                                "(the fp32 engine; the round's P-update GEMMs run on the tf32 tensor cores, three "
                                "products per term)")

    def capture(self):
        self.dbf.factorize(self.W, *self.f, outer=1, workspace=self.ws, **FACT_SCHED)

    def step(self):
        self.dbf.factorize(self.W, *self.f, outer=1, workspace=self.ws, **FACT_SCHED)

    def footprint_per_step(self):
        return self.ws.numel() + 4 * self.N * self.M

    def line(self, ms_step, steps):
        r = roofline_obj(self, ms_step, None, measured_traffic(self.key))
        r["peak_source"] = self.alu_peak_source
        return {"workload": self.key, "value": round(1e3 / ms_step, 3), "unit": "rounds/s",
                "ms_per_step": round(ms_step, 3), "us_per_call": round(ms_step * 1e3, 1), "calls_per_step": 1,
                "tflop_per_round": round(self.flops_per_call / 1e12, 4), "roofline": r}


QKV_SHAPES = ((4096, 4096, 3072), (1024, 4096, 1536), (1024, 4096, 2048))


class GroupedWorkload:
    """q, k and v of a 4096-wide block with grouped-query heads, each at its own middle dimension
    (non-uniform R), applied to the same tokens: one dbf_matmul_grouped call per group (or, with
    separate=True, three dbf_matmul calls), L groups with distinct factors per step."""

    def __init__(self, dbf, key, T, separate=False, max_calls=4096):
        import torch
        self.dbf, self.key, self.T, self.separate = dbf, key, T, separate
        base = []
        for k, (N, M, R) in enumerate(QKV_SHAPES):
            f = G.make_factors(N, M, R, 1, 6000 + k)
            base.append(to_device_factors(dbf, f))
            del f
        fp = sum(call_footprint(N, M, R, 1, T, pf.B1w.shape[1], pf.B2w.shape[1])
                 for (N, M, R), pf in zip(QKV_SHAPES, base))
        self.L = int(min(max_calls, max(8, math.ceil(4 * L2_BYTES / fp))))
        self.fp_call = fp
        x0 = bf16_dev(G.make_x(T, 4096, 6010))
        self.groups = [base] + [[clone_factors(dbf, pf) for pf in base] for _ in range(self.L - 1)]
        self.x = [x0] + [x0.clone() for _ in range(self.L - 1)]
        self.y = [[torch.empty((T, N), dtype=torch.bfloat16, device="cuda") for (N, _, _) in QKV_SHAPES]
                  for _ in range(self.L)]
        if separate:
            self.ws = dbf.new_workspace(max(dbf.workspace_bytes(pf, T) for pf in base), "cuda")
            self.launches_per_call = sum(dbf.launch_count(pf, T) for pf in base)
        else:
            self.ws = dbf.new_workspace(dbf.grouped_workspace_bytes(base, T), "cuda")
            self.launches_per_call = dbf.grouped_launch_count(base, T)
        self.bytes_per_call = sum(CFG.algorithmic_bytes(N, M, R, 1, T) for (N, M, R) in QKV_SHAPES)
        self.flops_per_call = sum(CFG.flops(N, M, R, 1, T) for (N, M, R) in QKV_SHAPES)
        self.bound = "hbm"
        self.graph = None

    def run_eager(self):
        for l in range(self.L):
            self.call_one(l)

    def call_one(self, l):
        x = self.x[l]
        if self.separate:
            for pf, y in zip(self.groups[l], self.y[l]):
                self.dbf.matmul(pf, x, y, workspace=self.ws)
        else:
            self.dbf.matmul_grouped(self.groups[l], [x, x, x], self.y[l], workspace=self.ws)

    capture = DecodeWorkload.capture
    step = DecodeWorkload.step

    def footprint_per_step(self):
        return self.L * self.fp_call

    @property
    def calls(self):
        return self.L

    @property
    def tokens_per_step(self):
        return self.L * self.T


class SegmentedWorkload:
    """Routed multi-adapter batches: one dbf_matmul_segmented call per adapter pool, L pools per step."""

    def __init__(self, dbf, key, w, max_calls=512):
        import torch
        self.dbf, self.key = dbf, key
        self.T = w.tokens[0]
        p0 = w.projections[0]
        self.N, self.M, self.R, self.ell = p0.N, p0.M, p0.R, p0.ell
        adapters = [to_device_factors(dbf, G.make_factors(p.N, p.M, p.R, p.ell, p.seed)) for p in w.projections]
        off, ad, _ = G.make_routing(self.T, w.n_adapters, w.routing_seed)
        touched = sorted(set(int(a) for a in ad))
        self.S = len(ad)
        ldw1, ldw2 = adapters[0].B1w.shape[1], adapters[0].B2w.shape[1]
        pool = len(adapters) * (self.N * ldw1 * 4 + self.R * ldw2 * 4 + 2 * self.ell * (self.N + self.R + self.M))
        fp = pool + 2 * self.T * (self.M + self.N)
        self.L = int(min(max_calls, max(4, math.ceil(4 * L2_BYTES / fp))))
        self.pools = []
        for l in range(self.L):
            ads = adapters if l == 0 else [clone_factors(dbf, a) for a in adapters]
            self.pools.append((ads, dbf.adapter_table(ads, "cuda")))
        self.off = torch.from_numpy(off).cuda()
        self.ad = torch.from_numpy(ad).cuda()
        x0 = bf16_dev(G.make_x(self.T, self.M, w.routing_seed))
        self.x = [x0] + [x0.clone() for _ in range(self.L - 1)]
        self.y = [torch.zeros((self.T, self.N), dtype=torch.bfloat16, device="cuda") for _ in range(self.L)]
        self.ws = dbf.new_workspace(dbf.segmented_workspace_bytes(self.N, self.M, self.R, self.ell, self.T, self.S),
                                    "cuda")
        self.launches_per_call = dbf.segmented_launch_count(self.N, self.M, self.R, self.ell, self.T, self.S)
        self.fp_call = fp
        # bytes: the sign bits and scales of every adapter the batch touches, plus x and y
        per_adapter = (self.R * (self.N + self.M)) // 8 + 2 * self.ell * (self.N + self.R + self.M)
        self.bytes_per_call = len(touched) * per_adapter + 2 * self.T * (self.M + self.N)
        self.flops_per_call = CFG.flops(self.N, self.M, self.R, self.ell, self.T)
        self.bound = "hbm"
        self.graph = None

    def run_eager(self):
        for l in range(self.L):
            self.call_one(l)

    def call_one(self, l):
        ads, table = self.pools[l]
        self.dbf.matmul_segmented(table, len(ads), self.N, self.M, self.R, self.ell, self.x[l], self.off,
                                  self.ad, self.y[l], workspace=self.ws)

    def footprint_per_step(self):
        return self.L * self.fp_call

    capture = DecodeWorkload.capture
    step = DecodeWorkload.step

    @property
    def calls(self):
        return self.L

    @property
    def tokens_per_step(self):
        return self.L * self.T


def time_steps(wl, steps, warmup, dist_mod=None, sampler=None):
    import torch
    for _ in range(warmup):
        wl.step()
    torch.cuda.synchronize()
    if dist_mod is not None:
        dist_mod.barrier()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    ctx = sampler if sampler is not None else _Null()
    with ctx:
        e0.record(stream)
        for _ in range(steps):
            wl.step()
        e1.record(stream)
        torch.cuda.synchronize()
    if dist_mod is not None:
        dist_mod.barrier()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1)


class _Null:
    def __enter__(self):
        return self

    def __exit__(self, *a):
        return False


def roofline_obj(wl, ms_per_call, peaks, traffic):
    if wl.bound == "hbm":
        achieved = wl.bytes_per_call / (ms_per_call * 1e-3) / 1e9
        peak = peaks["hbm_gbs"]
        unit = "GB/s"
    elif wl.bound == "alu":
        achieved = wl.flops_per_call / (ms_per_call * 1e-3) / 1e12
        peak = round(wl.alu_peak_tflops, 2)
        unit = "TFLOP/s"
    else:
        achieved = wl.flops_per_call / (ms_per_call * 1e-3) / 1e12
        peak = peaks["bf16_tflops"]
        unit = "TFLOP/s"
    d = {"bound": wl.bound, "achieved": round(achieved, 3), "peak": peak, "unit": unit,
         "frac": round(achieved / peak, 4), "traffic": traffic}
    if wl.bound == "tensor":
        d["frac_of_sustained"] = round(achieved / peaks["bf16_tflops_sustained"], 4)
    return d


# --------------------------------------------------------------- e2e (host io)

def measure_e2e(dbf, wl, steps):
    """Same calls through the host-io entry point (dbf_matmul_hostio_batch, one call per step): pinned
    host x in, host y out, copies inside the timed region."""
    import torch
    T, M, N = wl.T, wl.M, wl.N
    xh_all = torch.empty((wl.L, T, M), dtype=torch.bfloat16, pin_memory=True)
    yh_all = torch.empty((wl.L, T, N), dtype=torch.bfloat16, pin_memory=True)
    xh = [xh_all[l] for l in range(wl.L)]
    yh = [yh_all[l] for l in range(wl.L)]
    x_host = wl.x[0].cpu()
    for l in range(wl.L):
        xh[l].copy_(x_host)
    ws = dbf.new_workspace(dbf.hostio_batch_workspace_bytes(wl.factors, T), "cuda")

    def one_step(stream=None):
        # the step's L calls in one pipelined host-io call: copies overlap the kernels
        dbf.matmul_hostio_batch(wl.factors, xh, yh, workspace=ws, stream=stream)

    one_step()
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        one_step(s)
    torch.cuda.synchronize()
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    return {"value": round(wl.tokens_per_step / (ms * 1e-3), 1), "unit": "tokens/s",
            "h2d_bytes_per_step": wl.L * T * M * 2, "d2h_bytes_per_step": wl.L * T * N * 2,
            "ms_per_step": round(ms, 4),
            "path": "dbf_matmul_hostio_batch (pinned host x and y, the step's calls pipelined)"}


# ------------------------------------------------ single-call latency, cold L2

SINGLE_CALLS = 50


def measure_single_call(wl, peaks, calls=SINGLE_CALLS, reps=5):
    """Latency of one call with nothing of it in L2.  Two CUDA graphs are replayed: one holds
    `calls` x [write a buffer of twice the L2 size, one call] (so every input of every call
    comes from HBM), the other the same writes alone; the difference of their device times
    (CUDA events), divided by `calls`, is the cold latency of one call -- the device's event
    timer ticks in ~1 us steps, too coarse for a single call.  Median over `reps` replays."""
    import torch
    flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device="cuda")
    graphs = []
    for with_call in (True, False):
        for i in range(min(calls, wl.L)):  # eager warm-up of every call the graph holds
            if with_call:
                wl.call_one(i % wl.L)
        torch.cuda.synchronize()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for i in range(calls):
                flush.fill_(i & 0xFF)
                if with_call:
                    wl.call_one(i % wl.L)
        torch.cuda.synchronize()
        graphs.append(g)
    per = []
    for _ in range(reps + 1):
        t = []
        for g in graphs:
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            g.replay()
            e1.record()
            torch.cuda.synchronize()
            t.append(e0.elapsed_time(e1))
        per.append((t[0] - t[1]) / calls)
    del graphs, flush
    torch.cuda.empty_cache()
    ms = statistics.median(per[1:])
    r = roofline_obj(wl, ms, peaks, None)
    return {"protocol": f"cold L2: {2 * L2_BYTES // (1 << 20)} MiB written before each call; device time of "
                        f"{calls} x (write + call) minus {calls} x (write), per call, median of {reps} graph replays",
            "us_per_call": round(ms * 1e3, 3), "tokens_per_s": round(wl.T / (ms * 1e-3), 1),
            "roofline_frac": r["frac"], "roofline_achieved": r["achieved"], "roofline_unit": r["unit"]}


# ----------------------------------------------------------- CPU oracle timing

def oracle_threads():
    try:
        from threadpoolctl import threadpool_info
        import numpy  # noqa: F401
        info = threadpool_info()
        return max([i.get("num_threads", 1) for i in info] or [1])
    except Exception:
        return os.cpu_count() or 1


def time_oracle(seconds=10.0, min_calls=2):
    """The fp64 oracle as it stands on the headline workload: calls per bounded time."""
    from oracle import dbf_oracle as O
    p = CFG.ADAPTER_4K.projections[0]
    T = 16
    f = G.make_factors(p.N, p.M, p.R, p.ell, p.seed, p.sign_mode, p.scale_mode)
    xb = G.make_x(T, p.M, p.seed)
    O.matmul(xb, f)  # warm
    n = 0
    t0 = time.perf_counter()
    while n < min_calls or time.perf_counter() - t0 < seconds:
        O.matmul(xb, f)
        n += 1
    el = time.perf_counter() - t0
    return {"value": round(n * T / el, 2), "unit": "tokens/s", "cores": oracle_threads(), "kind": "oracle",
            "sample": f"{n} oracle calls (fp64 numpy, factored route) on one N=M=4096 R=64 ell=1 factor set, "
                      f"T={T} tokens each, {el:.1f} s"}


def _timed(fn, seconds, min_calls=1, max_calls=1000):
    fn()  # warm
    n = 0
    t0 = time.perf_counter()
    while n < min_calls or (time.perf_counter() - t0 < seconds and n < max_calls):
        fn()
        n += 1
    return n, time.perf_counter() - t0


def time_oracle_workload(key, seconds=2.0):
    """The fp64 oracle as it stands on one workload, on the host cores: the factored route
    (y_factored, what the library computes) for every workload, and the dense route (dW built,
    then x dW^T) for the three single-projection decode workloads; the MLP in prefill on a
    seeded 64-token subset (one call per projection); the routed batch as one call of the
    segmented oracle.  Returns {"factored": ..., "dense": ...} of cpu_baseline objects."""
    from oracle import dbf_oracle as O
    cores = oracle_threads()
    name, _, tok = key.rpartition("_T")
    T = int(tok) if tok.isdigit() else 0
    if name == "dbf1p5_one":
        name = "dbf1p5"  # the same product, one launch instead of two
    out = {}

    def obj(tokens, n, el, route, sample):
        return {"value": round(tokens * n / el, 2), "unit": "tokens/s", "cores": cores, "kind": "oracle",
                "route": route, "sample": f"{n} oracle calls (fp64 numpy), {sample}, {el:.2f} s"}

    if name in ("adapter4k", "dbf1p5", "tiny", "adapter4k_dx"):
        w = {"adapter4k": CFG.ADAPTER_4K, "adapter4k_dx": CFG.ADAPTER_4K, "dbf1p5": CFG.DBF_1P5,
             "tiny": CFG.TINY}[name]
        p = w.projections[0]
        f = G.make_factors(p.N, p.M, p.R, p.ell, p.seed, p.sign_mode, p.scale_mode)
        if name == "adapter4k_dx":
            dyb = G.make_x(T, p.N, p.seed + 7)
            n, el = _timed(lambda: O.matmul_dx(dyb, f), seconds)
            out["factored"] = obj(T, n, el, "factored (dx = dy dW)", f"{key}, T={T}")
            return out
        xb = G.make_x(T, p.M, p.seed, outlier_scale=w.outlier_scale)
        n, el = _timed(lambda: O.matmul(xb, f), seconds)
        out["factored"] = obj(T, n, el, "factored", f"{key}, T={T}")
        x64 = O.bf16_bits_to_f64(xb)
        n, el = _timed(lambda: O.round_to_bf16_bits(O.y_dense(x64, f)), seconds, max_calls=50)
        out["dense"] = obj(T, n, el, "dense (dW = sum_i diag(alpha_i) B1 diag(beta_i) B2 diag(gamma_i), "
                                     "then x dW^T)", f"{key}, T={T}")
        return out
    if name == "multiadapter":
        w = CFG.MULTI_ADAPTER
        fs = [G.make_factors(p.N, p.M, p.R, p.ell, p.seed) for p in w.projections]
        off, ad, _ = G.make_routing(w.tokens[0], w.n_adapters, w.routing_seed)
        xb = G.make_x(w.tokens[0], fs[0].B2.shape[1], w.routing_seed)
        n, el = _timed(lambda: O.matmul_segmented(xb, fs, off, ad), seconds)
        out["factored"] = obj(w.tokens[0], n, el, "factored, per segment", f"{key}, {len(ad)} segments")
        return out
    if name in ("dbfmlp", "dbfmlp_dx"):
        sub = 64
        tot_n, tot_el = 0, 0.0
        for p in CFG.DBF_MLP.projections:
            f = G.make_factors(p.N, p.M, p.R, p.ell, p.seed)
            if name == "dbfmlp":
                xb = G.make_x(sub, p.M, p.seed)
                n, el = _timed(lambda: O.matmul(xb, f), 0.0)
            else:
                dyb = G.make_x(sub, p.N, p.seed + 7)
                n, el = _timed(lambda: O.matmul_dx(dyb, f), 0.0)
            tot_n, tot_el = n, tot_el + el / n
            del f
        # tokens/s of one call per projection, as the GPU line counts them
        out["factored"] = {"value": round(sub * 2 / tot_el, 2), "unit": "tokens/s", "cores": cores,
                           "kind": "oracle", "route": "factored" + (" (dx = dy dW)" if name == "dbfmlp_dx" else ""),
                           "sample": f"seeded {sub}-token subset of the 2048 tokens (first {sub} rows of the "
                                     f"same draw), one oracle call per projection, {tot_el:.2f} s"}
        return out
    if name in ("dbfqkv", "dbfqkv_sep"):
        fs = [G.make_factors(N, M, R, 1, 6000 + k) for k, (N, M, R) in enumerate(QKV_SHAPES)]
        xb = G.make_x(T, 4096, 6010)
        n, el = _timed(lambda: O.matmul_grouped([xb, xb, xb], fs), seconds)
        out["factored"] = obj(T, n, el, "factored, three projections", f"{key}, T={T}")
        return out
    return out


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    from oracle import dbf_oracle as O
    p = CFG.ADAPTER_4K.projections[0]
    T = 16
    f = G.make_factors(p.N, p.M, p.R, p.ell, p.seed, p.sign_mode, p.scale_mode)
    xb = G.make_x(T, p.M, p.seed)
    for _ in range(args.warmup):
        O.matmul(xb, f)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        O.matmul(xb, f)
    el = time.perf_counter() - t0
    value = args.steps * T / el
    cores = oracle_threads()
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 2), "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(el * 1e3 / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "adapter4k: LoRDBA adapter branch N=M=4096 R=64 ell=1, T=16 decode tokens",
                   "tokens_per_call": T, "calls_per_step": 1, "l2": "not applicable (CPU)"},
        "cpu_baseline": {"value": round(value, 2), "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"{args.steps} timed oracle calls (fp64 numpy) of the headline workload, "
                                   f"one call per step"},
        "e2e": {"value": round(value, 2), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


# ----------------------------------------------------------------------- main

def workload_line(wl, ms_step, steps, peaks, extra=None):
    ms_call = ms_step / wl.calls
    d = {"workload": wl.key, "value": round(wl.tokens_per_step / (ms_step * 1e-3), 1), "unit": "tokens/s",
         "ms_per_step": round(ms_step, 4), "us_per_call": round(ms_call * 1e3, 3), "calls_per_step": wl.calls,
         "tokens_per_call": wl.T, "roofline": roofline_obj(wl, ms_call, peaks, measured_traffic(wl.key))}
    if extra:
        d.update(extra)
    return d


def make_workload(dbf, key, max_calls=None):
    """Workload by key: adapter4k_T{1,4,16}, dbf1p5_T{1,8}, dbf1p5_one_T8, tiny_T{1,8}, multiadapter_T256, dbfmlp_T2048,
    adapter4k_dx_T16, dbfmlp_dx_T2048, dbfmlp_bwd_T2048, dbfqkv_T8 (grouped), dbfqkv_sep_T8."""
    if key == "dbffact1p5":
        return FactorizeWorkload(dbf, key)
    cap = {} if max_calls is None else {"max_calls": max_calls}
    name, _, tok = key.rpartition("_T")
    T = int(tok)
    if name == "adapter4k_dx":
        return DecodeWorkload(dbf, key, CFG.ADAPTER_4K.projections[0], T, transposed=True, **cap)
    if name == "dbfmlp_dx":
        return PrefillWorkload(dbf, key, CFG.DBF_MLP.projections, T, transposed=True)
    if name == "dbfmlp_bwd":
        return BackwardWorkload(dbf, key, CFG.DBF_MLP.projections, T)
    if name == "dbfqkv":
        return GroupedWorkload(dbf, key, T, **cap)
    if name == "dbfqkv_sep":
        return GroupedWorkload(dbf, key, T, separate=True, **cap)
    if name == "adapter4k":
        return DecodeWorkload(dbf, key, CFG.ADAPTER_4K.projections[0], T, **cap)
    if name == "dbf1p5":
        return DecodeWorkload(dbf, key, CFG.DBF_1P5.projections[0], T, outlier_scale=CFG.DBF_1P5.outlier_scale,
                              **cap)
    if name == "dbf1p5_one":
        return DecodeWorkload(dbf, key, CFG.DBF_1P5.projections[0], T, outlier_scale=CFG.DBF_1P5.outlier_scale,
                              one_launch=True, **cap)
    if name == "tiny":
        return DecodeWorkload(dbf, key, CFG.TINY.projections[0], T, **cap)
    if name == "multiadapter":
        return SegmentedWorkload(dbf, key, CFG.MULTI_ADAPTER, **cap)
    if name == "dbfmlp":
        return PrefillWorkload(dbf, key, CFG.DBF_MLP.projections, T)
    raise ValueError(f"unknown workload {key!r}")


WORKLOAD_TITLES = {
    "adapter4k": "adapter4k: LoRDBA adapter branch N=M=4096 R=64 ell=1, T={T} decode tokens",
    "dbf1p5": "dbf1p5: DBF 1.5 bits/weight N=M=4096 R=3072 ell=1, 1% outlier columns x20, T={T} decode tokens",
    "dbf1p5_one": "dbf1p5_one: the dbf1p5 decode with both stages in one cooperative launch (grid-wide "
                  "barrier between them), the comparison arm of the two-launch form, T={T} decode tokens",
    "tiny": "tiny: N=M=256 R=32 ell=1, T={T} tokens",
    "multiadapter": "multiadapter: 64 adapters N=M=4096 R=32 ell=2, T={T} routed decode tokens",
    "dbfmlp": "dbfmlp: DBF MLP up 14336x4096 + down 4096x14336, R=5013 ell=2, T={T} prefill tokens",
    "adapter4k_dx": "adapter4k_dx: backward dx = dy dW of the LoRDBA adapter branch N=M=4096 R=64 ell=1, T={T}",
    "dbfmlp_dx": "dbfmlp_dx: backward dx = dy dW of the DBF MLP up + down projections, R=5013 ell=2, T={T}",
    "dbfmlp_bwd": "dbfmlp_bwd: backward pass (dx, dalpha, dbeta, dgamma) of the DBF MLP up + down projections, "
                  "R=5013 ell=2, T={T}",
    "dbfqkv": "dbfqkv: q 4096x4096 R=3072, k and v 1024x4096 R=1536 / 2048 (non-uniform R), ell=1, one grouped "
              "call per token batch, T={T} decode tokens",
    "dbfqkv_sep": "dbfqkv_sep: the same q, k, v projections as three separate calls, T={T} decode tokens",
    "dbffact1p5": "dbffact1p5: double binary factorization of a dense 4096x4096 fp32 weight at k=3072 "
                  "(1.5 bits/weight), one alternating round (A-step + B-step, 10 ADMM iterations each, "
                  "8 power iterations per SVID)",
}

SECONDARY = ["adapter4k_T1", "adapter4k_T4", "dbf1p5_T1", "dbf1p5_T8", "dbf1p5_one_T8", "tiny_T8", "multiadapter_T256",
             "dbfmlp_T2048", "adapter4k_dx_T16", "dbfmlp_dx_T2048", "dbfmlp_bwd_T2048", "dbfqkv_T8",
             "dbfqkv_sep_T8", "dbffact1p5"]


def main(argv=None):
    args = parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)

    import torch
    rank, world, local = dist_env()
    dist_mod = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
        dist_mod = dist
    else:
        torch.cuda.set_device(0)

    from double_binary_rank_packed_b300 import build
    build.build()
    from double_binary_rank_packed_b300 import dbf

    peaks, peak_src = load_peaks()

    # ---------------- main line (default: the headline adapter4k, T = 16), streamed
    head = make_workload(dbf, args.workload, args.max_calls)
    head.capture()
    sampler = ClockSampler(local)
    ms = time_steps(head, args.steps, args.warmup, dist_mod, sampler)
    ms_max, tok_total = aggregate(ms, head.tokens_per_step * args.steps, dist_mod)
    ms_step = ms_max / args.steps
    value = tok_total / (ms_max * 1e-3)
    ms_call = ms_step / head.calls
    clocks = sampler.summary()
    rl = roofline_obj(head, ms_call, peaks, measured_traffic(head.key))
    rl["peak_source"] = peak_src
    rl["per"] = "call"
    rl["us_per_call"] = round(ms_call * 1e3, 3)

    name, _, tok = head.key.rpartition("_T")
    footprint = head.footprint_per_step()
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16",
        "arith": "fp16 tensor-core operands (+-1 signs, gamma*x, beta*u), fp32 accumulation, bf16 in/out",
        "data": "synthetic",
        "config": {"workload": WORKLOAD_TITLES[name].format(T=tok),
                   "tokens_per_call": head.T, "calls_per_step": head.calls,
                   "distinct_factor_sets_per_step": head.calls,
                   "l2": ("no flush: each step touches %.0f MB of distinct inputs (%s 4x the 126 MB L2)"
                          % (footprint / 1e6, ">" if footprint > 4 * L2_BYTES else "NOT >")),
                   "launch": "one CUDA graph per step, programmatic dependent launch between kernels",
                   "parallelism": f"replicas x{world} (independent projections per rank)"},
        "roofline": rl,
        "clocks": clocks,
        "gpu_launches": args.steps * head.calls * head.launches_per_call,
    }

    if rank == 0 and not args.no_e2e and isinstance(head, DecodeWorkload):
        line["e2e"] = measure_e2e(dbf, head, max(3, min(args.steps, 10)))
    if rank == 0 and hasattr(head, "call_one") and not args.no_single:
        line["single_call"] = measure_single_call(head, peaks)
        line["roofline"]["protocol"] = "streamed: one CUDA graph of distinct calls, PDL, per-call = step / calls"
    if rank == 0 and world == 1 and not args.no_cpu:
        line["cpu_baseline"] = time_oracle()
        extra = time_oracle_workload(head.key)
        if "dense" in extra:
            line["cpu_baseline_dense"] = extra["dense"]

    if world == 1 and not args.no_also:
        also = []
        for key in SECONDARY:
            if key == head.key or (args.only and key != args.only):
                continue
            wl = make_workload(dbf, key)
            wl.capture()
            s2 = ClockSampler(local)
            if isinstance(wl, FactorizeWorkload):
                fsteps = max(3, min(args.steps, 5))
                ms_w = time_steps(wl, fsteps, 3, None, s2)
                d = wl.line(ms_w / fsteps, fsteps)
                d["gpu_launches"] = fsteps * wl.launches_per_call
                d["clocks"] = s2.summary()
                also.append(d)
                del wl
                torch.cuda.empty_cache()
                continue
            ms_w = time_steps(wl, args.steps, args.warmup, None, s2)
            d = workload_line(wl, ms_w / args.steps, args.steps, peaks)
            d["clocks"] = s2.summary()
            d["gpu_launches"] = args.steps * wl.calls * wl.launches_per_call
            if hasattr(wl, "call_one") and not args.no_single:
                d["single_call"] = measure_single_call(wl, peaks)
            if not args.no_cpu:
                cb = time_oracle_workload(key)
                if "factored" in cb:
                    d["cpu_baseline"] = cb["factored"]
                if "dense" in cb:
                    d["cpu_baseline_dense"] = cb["dense"]
            also.append(d)
            del wl
            torch.cuda.empty_cache()
        line["also"] = also

    if rank == 0:
        print(json.dumps(line))
    if dist_mod is not None:
        dist_mod.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
