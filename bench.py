"""Benchmark of the fused FlashAdamW step on the Llama-3-8B tensor list.

One step = one ``fo_adamw_step`` call (one kernel launch) over all 291
parameter tensors (8,030,261,248 parameters): bf16 theta' + int8 rho (24-bit
master), int8 / uint8 m and v codes with fp16 group-32 scales, bf16 grads.
Inputs are synthetic (seeded N(0, 0.02) weights, N(0, 1e-3) grads) and far
larger than L2 (98 GB move per step), so no L2 flush is needed.

Prints ONE JSON line (rank 0).  ``--impl reference`` times the CPU oracle
instead (the slow, literal CPU statement of the method) on a bounded sample of
the same workload.
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time
from concurrent.futures import ThreadPoolExecutor

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads as W  # noqa: E402

METRIC = "params/s and achieved HBM GB/s (% of GB300 peak) for fused AdamW step"
UNIT = "params/s"
# The workload: the Llama-3-8B list (24-bit master, int8 rho; the headline) or
# the 1.1B list (32-bit master, int16 rho), chosen with --workload.
WORKLOADS = {
    W.LLAMA3_8B.name: (W.LLAMA3_8B, W.LLAMA3_8B_HYPER, W.LLAMA3_8B_MASTER_BITS),
    W.TINYLLAMA_1B.name: (W.TINYLLAMA_1B, W.TINYLLAMA_HYPER, W.TINYLLAMA_MASTER_BITS),
}
SINGLE = "single-65553"
MODEL = W.LLAMA3_8B
HYPER = W.LLAMA3_8B_HYPER
MASTER_BITS = W.LLAMA3_8B_MASTER_BITS
RHO_BITS = 8 if MASTER_BITS == 24 else 16


def use_workload(name: str) -> None:
    """Select the tensor list, hyper-parameters and master width of a workload."""
    global MODEL, HYPER, MASTER_BITS, RHO_BITS
    MODEL, HYPER, MASTER_BITS = WORKLOADS[name]
    RHO_BITS = 8 if MASTER_BITS == 24 else 16
FALLBACK_HBM_GBS = 6800.0


def workload_config(numels) -> dict:
    return {
        "workload": (f"{MODEL.name} tensor list: {len(numels)} tensors, {sum(numels):,} params; "
                     f"bf16 theta' + int{RHO_BITS} rho ({MASTER_BITS}-bit master), int8/uint8 m/v codes "
                     f"+ fp16 group-32 scales, bf16 grads; lr {HYPER.lr:g}, betas ({HYPER.beta1:g}, "
                     f"{HYPER.beta2:g}), eps {HYPER.eps:g}, wd {HYPER.weight_decay:g}"),
        "params": int(sum(numels)),
        "tensors": len(numels),
        "l2": "inputs larger than L2 (no flush needed)",
    }


def algorithmic_bytes(numels, grad_bytes=2, rho_bytes=None) -> int:
    """Bytes the step must move: read grad, theta', rho, m/v codes and scales;
    write theta', rho, m/v codes and scales (12.25 B/param for bf16 grad + int8 rho)."""
    if rho_bytes is None:
        rho_bytes = RHO_BITS // 8
    total = 0
    for n in numels:
        g = (n + 31) // 32
        total += n * (grad_bytes + 2 * 2 + 2 * rho_bytes + 2 * 1 + 2 * 1) + 2 * 2 * (2 * g)
    return total


# DRAM traffic of the pipelined kernel, from one ncu capture each
# (dram__bytes_read.sum + dram__bytes_write.sum of one launch over the
# parameters of decoder layer 0, bf16 grads), keyed by (kernel, format, rho
# width) and valid only for the kernel sources they were taken on.  A capture
# on one layer reads up to one L2's worth less than the algorithmic bytes (the
# previous launch's last tiles are still in L2); that saving is bounded by the
# L2 size, not proportional to the launch, so it is subtracted once, not
# scaled: a full launch moves (capture + saving) * n / n_capture - saving.
L2_BYTES = 126 * 2**20
_CAPTURE_SOURCES = {
    "quantized_state_optimizer_gb300/csrc/fo_step.cu": "7763e84c6e2c76f2a38afd4fd8a7456b1bfe1532987d74ada1c0cf0a38e5821b",
    "quantized_state_optimizer_gb300/csrc/fo_device.cuh": "0f67b3354cfa65905708fe4d4c4bf24a285c2c36db7f160db62129242a2f1373",
}
# (kernel, format, rho bits) -> (read bytes, write bytes, parameters, algorithmic bytes per parameter)
TRAFFIC_CAPTURE: dict = {
    # 8B list, layer 0 (9 tensors), int8 rho
    ("fo::adamw_step_kernel", None, 8): (1_565_242_000, 1_074_010_000, 218_112_000, 12.25),
    # 1.1B list, layer 0 (9 tensors), int16 rho
    ("fo::adamw_step_kernel", None, 16): (361_392_384, 215_593_984, 44_044_288, 14.25),
}


def captured_traffic(n_params: int, kernel: str = "fo::adamw_step_kernel", fmt: str | None = None,
                     rho_bits: int | None = None) -> float | None:
    """Per-launch DRAM traffic of a full launch over n_params, from the
    capture, or None when there is no capture for this kernel and format or
    the kernel changed since."""
    import hashlib
    cap = TRAFFIC_CAPTURE.get((kernel, fmt, RHO_BITS if rho_bits is None else rho_bits))
    if cap is None:
        return None
    for rel, digest in _CAPTURE_SOURCES.items():
        try:
            with open(os.path.join(ROOT, rel), "rb") as fh:
                if hashlib.sha256(fh.read()).hexdigest() != digest:
                    return None
        except OSError:
            return None
    read, write, n_cap, per_param = cap
    measured = read + write
    saving = min(max(0.0, per_param * n_cap - measured), float(L2_BYTES))
    return (measured + saving) * n_params / n_cap - saving


def load_peak() -> tuple[float, str]:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as fh:
            return float(json.load(fh)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# ------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.lines: list[str] = []
        ident = None
        try:
            ident = "GPU-" + str(torch.cuda.get_device_properties(device_index).uuid)
        except Exception:
            pass
        self.ident = ident if ident else str(device_index)

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.ident, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self._t.join(timeout=2)

    def summary(self) -> dict | None:
        rows = []
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                rows.append((float(parts[0]), float(parts[1]), parts[4:8]))
            except ValueError:
                continue
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i, v in enumerate(r) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------ GPU arm
def bench_specs(layers: int | None):
    """The full tensor list, or (for profiling captures that must stay small) only
    the tensors of the first ``layers`` decoder layers."""
    specs = W.llama_tensor_list(MODEL)
    if layers is None:
        return specs
    keep = tuple(f"layers.{i}." for i in range(layers))
    return [s for s in specs if s.name.startswith(keep)]


def build_state(device, layers: int | None = None, fmt: str | None = None, optimizer: str = "adamw"):
    """The state of the list (θ from the input recipe, zero states) with the
    gradients drawn for step 1 in its own grad slab, and the further
    gradient sets (``grad_sets(...)``) that the timed steps cycle through."""
    from quantized_state_optimizer_gb300.optim import FlashAdamWState
    specs = bench_specs(layers)
    numels = [s.numel for s in specs]
    if fmt is not None:
        st = GeneralState(numels, *fmt.split(":"), device, optimizer)
    else:
        st = FlashAdamWState(numels, rho_bits=RHO_BITS, grad_dtype=torch.bfloat16, device=device)
    wid = W.WORKLOAD_IDS[MODEL.name]
    for i, k in enumerate(tensor_indices(specs)):
        st.init_theta(i, W.init_theta(specs[i], wid, k, device))
        W.make_grad(specs[i].numel, wid, k, 1, device, out=st.grad_view(i))
    torch.cuda.synchronize()
    return st, numels


def tensor_indices(specs) -> list[int]:
    """Each tensor's index in the full list (the seeds follow it)."""
    all_specs = W.llama_tensor_list(MODEL)
    return [all_specs.index(s) for s in specs]


# Resident gradient sets the timed steps cycle through: step t reads the set
# drawn for step 1 + (t - 1) mod GRAD_SETS.  A gradient that never changes
# drives m and v towards values with few significant bits, which no training
# run sees; drawing a new one inside the timed region would time the input
# generator.
GRAD_SETS = 2


def grad_sets(st, layers: int | None, device) -> list[torch.Tensor]:
    """The grad slabs of steps 1..GRAD_SETS in the layout of ``st.grad``:
    ``st.grad`` itself (drawn by ``build_state``) and the later ones."""
    specs = bench_specs(layers)
    wid = W.WORKLOAD_IDS[MODEL.name]
    slabs = [st.grad]
    for step in range(2, GRAD_SETS + 1):
        slab = torch.zeros_like(st.grad)
        for i, k in enumerate(tensor_indices(specs)):
            v = st.grad_view(i)
            o = v.storage_offset() - st.grad.storage_offset()
            W.make_grad(specs[i].numel, wid, k, step, device, out=slab[o:o + v.numel()])
        slabs.append(slab)
    torch.cuda.synchronize()
    return slabs


class BenchSteps:
    """The timed step: step t launches over gradient set (t - 1) mod
    len(slabs).  By default one launch per step over every tensor.  With
    ``per_tensor`` it issues the step as gradient release launches it: one
    single-tensor ``fo_adamw_step`` launch per tensor of at least ``bucket``
    elements (what ``FlashAdamW(gradient_release=True)`` launches from each
    parameter's post-accumulate-grad hook) and one launch for all smaller
    tensors (its bucket of small parameters), here back to back on one
    stream."""

    def __init__(self, st, slabs, per_tensor: bool = False, bucket: int = 1 << 20):
        self.st = st
        self.general = isinstance(st, GeneralState)
        self.sets = []
        for slab in slabs:
            full = st.grad_array(slab) if self.general else st.fo_tensors(
                grads=[slab[st.grad_view(i).storage_offset() - st.grad.storage_offset():][:n]
                       for i, n in enumerate(st.numels)])
            if not per_tensor:
                self.sets.append([full])
                continue
            ctype = type(full[0])
            big = [i for i, n in enumerate(st.numels) if n >= bucket]
            small = [i for i, n in enumerate(st.numels) if n < bucket]
            arrs = [(ctype * 1)(full[i]) for i in big]
            if small:
                arrs.append((ctype * len(small))(*[full[i] for i in small]))
            self.sets.append(arrs)
        self.launches_per_step = len(self.sets[0])

    def step(self, t, lr, beta1, beta2, eps, weight_decay, stream=None) -> None:
        import quantized_state_optimizer_gb300 as fo
        for arr in self.sets[(t - 1) % len(self.sets)]:
            if self.general:
                self.st.launch(arr, t, lr, beta1, beta2, eps, weight_decay, stream)
            else:
                fo.fo_adamw_step(arr, self.st.grad_dtype, lr, beta1, beta2, eps, weight_decay, t,
                                 self.st.rho_bits, stream)


# ------------------------------------------------- the ablation formats
def general_bytes_per_param(pf: str, sf: str, optimizer: str = "adamw") -> float:
    """Algorithmic bytes of one step per parameter in a format (bf16 grads):
    AdamW reads and writes two states, SGD one (the momentum)."""
    param = 4 if pf == "f32" else 2
    rho = {"bf16_rho8": 1, "bf16_rho16": 2}.get(pf, 0)
    one_state = 8.0 if sf == "f32" else 2.0 + 2 * 2 / 32
    return 2 + 2 * param + 2 * rho + (2 if optimizer == "adamw" else 1) * one_state


def step_kernel_name(fmt: str | None, optimizer: str) -> str:
    """The kernel one step launches: the pipelined step kernel in every
    format (AdamW through fo_adamw_step or fo_adamw_step_general, SGD
    through fo_sgd_step)."""
    return "fo::sgd_step_kernel" if optimizer == "sgd" else "fo::adamw_step_kernel"


class GeneralState:
    """Flat device slabs of the list in one of the ablation formats, and the
    ``fo_tensor_general`` array over them (for ``fo_adamw_step_general``)."""

    def __init__(self, numels, pf: str, sf: str, device, optimizer: str = "adamw"):
        import quantized_state_optimizer_gb300 as fo
        self.pf, self.sf, self.optimizer = pf, sf, optimizer
        align = lambda n: (n + 15) // 16 * 16  # noqa: E731
        offs, o = [], 0
        for n in numels:
            offs.append(o)
            o += align(n)
        goffs, go = [], 0
        for n in numels:
            goffs.append(go)
            go += align((n + 31) // 32)
        total, gtotal = max(o, 16), max(go, 16)
        self.offs, self.numels = offs, numels
        self.param = torch.zeros(total, dtype=torch.float32 if pf == "f32" else torch.bfloat16, device=device)
        self.rho = (torch.zeros(total, dtype=torch.int8 if pf == "bf16_rho8" else torch.int16, device=device)
                    if pf in ("bf16_rho8", "bf16_rho16") else None)
        st_dt = (torch.float32, torch.float32) if sf == "f32" else (torch.int8, torch.uint8)
        self.m = torch.zeros(total, dtype=st_dt[0], device=device)
        self.v = torch.zeros(total, dtype=st_dt[1], device=device)
        self.ms = None if sf == "f32" else torch.zeros(gtotal, dtype=torch.float16, device=device)
        self.vs = None if sf == "f32" else torch.zeros(gtotal, dtype=torch.float16, device=device)
        self.grad = torch.zeros(total, dtype=torch.bfloat16, device=device)
        self.goffs = goffs
        self.arr = self.grad_array(self.grad)

    def grad_array(self, grad: torch.Tensor):
        """``fo_tensor_general`` array over the slabs, reading gradients from ``grad``."""
        import quantized_state_optimizer_gb300 as fo
        ptr = lambda t, off, esz: t.data_ptr() + off * esz if t is not None else None  # noqa: E731
        offs, goffs = self.offs, self.goffs
        return (fo.FoTensorGeneral * len(self.numels))(*[
            fo.FoTensorGeneral(ptr(self.param, offs[i], self.param.element_size()),
                               ptr(self.rho, offs[i], self.rho.element_size() if self.rho is not None else 0),
                               ptr(grad, offs[i], 2), ptr(self.m, offs[i], self.m.element_size()),
                               ptr(self.ms, goffs[i], 2), ptr(self.v, offs[i], self.v.element_size()),
                               ptr(self.vs, goffs[i], 2), n)
            for i, n in enumerate(self.numels)])

    def init_theta(self, i: int, theta: torch.Tensor) -> None:
        import quantized_state_optimizer_gb300 as fo
        o, n = self.offs[i], self.numels[i]
        if self.rho is not None:
            fo.fo_split(theta, 8 if self.pf == "bf16_rho8" else 16, self.param[o:o + n], self.rho[o:o + n])
        else:
            self.param[o:o + n].copy_(theta)

    def grad_view(self, i: int) -> torch.Tensor:
        return self.grad[self.offs[i]:self.offs[i] + self.numels[i]]

    def step(self, t, lr, beta1, beta2, eps, weight_decay, stream=None) -> None:
        self.launch(self.arr, t, lr, beta1, beta2, eps, weight_decay, stream)

    def launch(self, arr, t, lr, beta1, beta2, eps, weight_decay, stream=None) -> None:
        import quantized_state_optimizer_gb300 as fo
        if self.optimizer == "sgd":  # momentum beta1, the same lr and weight decay
            fo.fo_sgd_step(arr, self.pf, self.sf, torch.bfloat16, lr, beta1, weight_decay, stream)
        else:
            fo.fo_adamw_step_general(arr, self.pf, self.sf, torch.bfloat16, lr, beta1, beta2, eps,
                                     weight_decay, t, stream)


def time_steps(st, steps: int, warmup: int, stream, dist_on: bool) -> tuple[float, list[float]]:
    h = HYPER
    t = 0
    for _ in range(warmup):
        t += 1
        st.step(t, h.lr, h.beta1, h.beta2, h.eps, h.weight_decay, stream=stream)
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    if dist_on:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for k in range(steps):
        t += 1
        starts[k].record(stream)
        st.step(t, h.lr, h.beta1, h.beta2, h.eps, h.weight_decay, stream=stream)
        ends[k].record(stream)
    t1.record(stream)
    torch.cuda.synchronize()
    if dist_on:
        torch.distributed.barrier()
    total_ms = t0.elapsed_time(t1)
    per = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    return total_ms, per


def time_e2e(st, numels, steps: int, stream, slabs) -> dict:
    """Same step through the public API with host buffers: each step uploads the
    bf16 grads from pinned host memory and downloads the updated bf16
    parameters into pinned host memory (``FlashAdamWState.step_from_host``,
    which overlaps both copies with the step chunk by chunk), all inside the
    timed region.  The host holds the gradient sets of the device bench
    (``slabs``) and step t uploads set (t - 1) mod len(slabs)."""
    h = HYPER
    host_grads = []
    for slab in slabs:
        hg = torch.empty(slab.numel(), dtype=slab.dtype, pin_memory=True)
        hg.copy_(slab)
        host_grads.append(hg)
    host_param = torch.empty(st.param.numel(), dtype=st.param.dtype, pin_memory=True)
    torch.cuda.synchronize()
    # untimed: one step per host buffer, so that no buffer's first transfer
    # falls in the timed region
    t = 1000
    for _ in host_grads:
        st.step_from_host(t, h.lr, h.beta1, h.beta2, h.eps, h.weight_decay, host_grads[(t - 1) % len(host_grads)],
                          host_param, stream=stream)
        t += 1
    t -= 1
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    ev[0].record(stream)
    for k in range(steps):
        t += 1
        st.step_from_host(t, h.lr, h.beta1, h.beta2, h.eps, h.weight_decay, host_grads[(t - 1) % len(host_grads)],
                          host_param, stream=stream)
        ev[k + 1].record(stream)
    torch.cuda.synchronize()
    per = [ev[k].elapsed_time(ev[k + 1]) for k in range(steps)]
    ms = ev[0].elapsed_time(ev[steps]) / steps
    n = sum(numels)
    return {"value": n / (ms * 1e-3), "unit": UNIT, "ms_per_step": ms,
            "ms_per_step_min": min(per), "ms_per_step_median": statistics.median(per), "ms_per_step_max": max(per),
            "h2d_bytes_per_step": int(host_grads[0].numel() * host_grads[0].element_size()),
            "d2h_bytes_per_step": int(host_param.numel() * host_param.element_size()),
            "steps": steps, "api": "FlashAdamWState.step_from_host (8 chunks, copies overlapped)"}


def single_tensor_line(steps: int, warmup: int, device) -> dict:
    """The single-tensor workload: 65,553 parameters, fp32 grads (seed 1000 + t,
    the ten steps of the input recipe cycled), int8 rho, lr 1e-3, betas (0.9,
    0.999), eps 1e-8, wd 0.01.  Its 0.93 MB fit in L2, so one step is bound by
    launch and pipeline latency: no roofline claim."""
    from quantized_state_optimizer_gb300 import fo_adamw_step
    from quantized_state_optimizer_gb300.optim import FlashAdamWState
    n = W.SINGLE_TENSOR_NUMEL
    h = W.SINGLE_TENSOR_HYPER
    st = FlashAdamWState([n], rho_bits=8, grad_dtype=torch.float32, device=device)
    st.init_theta(0, W.single_tensor_theta(n).to(device))
    grads = [W.single_tensor_grad(t, n).to(device) for t in range(1, h.steps + 1)]
    arrs = [st.fo_tensors(grads=[g]) for g in grads]
    stream = torch.cuda.Stream(device=device)

    def step(t):
        fo_adamw_step(arrs[(t - 1) % len(arrs)], torch.float32, h.lr, h.beta1, h.beta2, h.eps, h.weight_decay, t, 8,
                      stream)

    t = 0
    for _ in range(warmup):
        t += 1
        step(t)
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    ev[0].record(stream)
    for k in range(steps):
        t += 1
        step(t)
        ev[k + 1].record(stream)
    torch.cuda.synchronize()
    per = [ev[k].elapsed_time(ev[k + 1]) for k in range(steps)]
    ms = ev[0].elapsed_time(ev[steps]) / steps
    return {"metric": METRIC, "value": n / (ms * 1e-3), "unit": UNIT, "n_gpus": 1, "steps": steps, "warmup": warmup,
            "ms_per_step": ms, "ms_per_step_median": statistics.median(per), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": (f"single tensor: {n:,} params, fp32 grads (ten seeded steps, cycled), bf16 "
                                    f"theta' + int8 rho (24-bit master), lr {h.lr:g}, betas ({h.beta1:g}, "
                                    f"{h.beta2:g}), eps {h.eps:g}, wd {h.weight_decay:g}"),
                       "params": n, "tensors": 1,
                       "l2": "0.93 MB fit in L2: latency-bound, no roofline claim",
                       "bytes_per_step": algorithmic_bytes([n], grad_bytes=4)},
            "roofline": None, "cpu_baseline": None, "e2e": None, "gpu_launches": steps}


# ------------------------------------------------------------ CPU oracle
def oracle_sample(total_params: int, chunk: int = 1 << 20, seed: int = 1, layers: int = 2):
    """A bounded, seeded sample of the workload for the CPU oracle: group-aligned
    chunks of the first decoder layers' tensors (each group is independent, so
    any group-aligned piece is a valid unit of the step)."""
    import oracle as O
    keep = tuple(f"layers.{i}." for i in range(layers))
    specs = [s for s in W.llama_tensor_list(MODEL) if s.name.startswith(keep)]
    pieces = []
    left = total_params
    gen = torch.Generator().manual_seed(seed)
    for s in specs:
        for off in range(0, s.numel, chunk):
            n = min(chunk, s.numel - off)
            if left <= 0:
                break
            n = min(n, left)
            theta = torch.ones(n) if s.is_norm else torch.randn(n, generator=gen) * 0.02
            g = (torch.randn(n, generator=gen) * 1e-3).to(torch.bfloat16)
            gb = g.view(torch.int16).numpy().view(np.uint16)
            pieces.append((O.TensorState.init(theta.numpy(), master_bits=MASTER_BITS), gb))
            left -= n
    return pieces


def run_oracle_steps(pieces, steps: int, threads: int, t0: int = 1) -> float:
    """Wall seconds for ``steps`` oracle steps over the sample (threads over pieces)."""
    import oracle as O
    h = HYPER

    def one(p, t):
        st, g = p
        O.adamw_step(st, g, t, h.lr, h.beta1, h.beta2, h.eps, h.weight_decay)

    start = time.perf_counter()
    with ThreadPoolExecutor(max_workers=threads) as ex:
        for k in range(steps):
            list(ex.map(lambda p: one(p, t0 + k), pieces))
    return time.perf_counter() - start


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def cpu_baseline(sample_params: int, steps: int) -> dict:
    cores = host_cores()
    pieces = oracle_sample(sample_params)
    n = sum(p[0].numel for p in pieces)
    run_oracle_steps(pieces, 1, cores)  # first touch
    sec = run_oracle_steps(pieces, steps, cores, t0=2)
    # one thread, one step over the first 8 pieces: the oracle's serial speed
    few = pieces[:8]
    sec1 = run_oracle_steps(few, 1, 1, t0=steps + 2)
    return {"value": n * steps / sec, "unit": UNIT, "cores": cores, "kind": "oracle",
            "seconds": sec, "single_thread_value": sum(p[0].numel for p in few) / sec1,
            "sample": (f"{n:,} params (decoder layers 0-1 of the {MODEL.name} list) in group-aligned "
                       f"1M-element pieces, {steps} steps, one thread per piece on {cores} host cores")}


# ------------------------------------------------------------ host link
def host_link(gib: int = 8) -> dict:
    """Pinned host <-> device copy bandwidth (GB/s) on 2*gib GB buffers, one
    direction at a time and both at once: the ceiling of the e2e number."""
    n = gib << 30
    h = torch.empty(n, dtype=torch.bfloat16, pin_memory=True)
    h2 = torch.empty(n, dtype=torch.bfloat16, pin_memory=True)
    d = torch.empty(n, dtype=torch.bfloat16, device="cuda")
    d2 = torch.empty(n, dtype=torch.bfloat16, device="cuda")
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()

    def timed(fn):
        torch.cuda.synchronize()
        t = time.perf_counter()
        fn()
        torch.cuda.synchronize()
        return time.perf_counter() - t

    def both():
        with torch.cuda.stream(s1):
            d.copy_(h, non_blocking=True)
        with torch.cuda.stream(s2):
            h2.copy_(d2, non_blocking=True)

    timed(lambda: d.copy_(h, non_blocking=True))
    gb = n * 2 / 1e9
    return {"h2d_gbs": gb / timed(lambda: d.copy_(h, non_blocking=True)),
            "d2h_gbs": gb / timed(lambda: h2.copy_(d, non_blocking=True)),
            "both_directions_gbs": 2 * gb / timed(both), "bytes_each": int(n * 2)}


# --------------------------------------------------- standalone kernels
def pair_kernels(n: int = 1 << 30, reps: int = 5) -> dict:
    """The standalone kernels on ``n`` fp32 elements (far above L2): fo_quantize
    and fo_dequantize in all four specs, fo_split and fo_reconstruct for both
    rho widths.  Per kernel: the mean launch time over ``reps`` launches (CUDA
    events on the launching stream, after two warm-up launches) and its
    algorithmic bytes per launch against the measured copy bandwidth."""
    import quantized_state_optimizer_gb300 as fo
    peak, src = load_peak()
    dev = torch.device("cuda")
    ng = (n + 31) // 32
    gen = torch.Generator(device=dev).manual_seed(5)
    x = torch.randn(n, device=dev, generator=gen) * 1e-3
    out = torch.empty(n, device=dev)
    codes = {True: torch.empty(n, dtype=torch.int8, device=dev), False: torch.empty(n, dtype=torch.uint8, device=dev)}
    scales = torch.empty(ng, dtype=torch.float16, device=dev)
    theta_bf = torch.empty(n, dtype=torch.bfloat16, device=dev)
    rhos = {8: torch.empty(n, dtype=torch.int8, device=dev), 16: torch.empty(n, dtype=torch.int16, device=dev)}
    stream = torch.cuda.Stream()

    def timed(fn) -> float:
        with torch.cuda.stream(stream):  # torch ops too run on the timed stream
            for _ in range(2):
                fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        with torch.cuda.stream(stream):
            for _ in range(reps):
                fn()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / reps

    rows = []

    def add(kernel, variant, ms, nbytes):
        gbs = nbytes / (ms * 1e-3) / 1e9
        rows.append({"kernel": kernel, "variant": variant, "ms": ms, "bytes": nbytes, "gbs": gbs,
                     "frac": gbs / peak})

    for spec in ("momentum", "variance", "momentum_linear", "variance_linear"):
        signed = spec.startswith("momentum")
        src_x = x if signed else x.abs()  # the variance specs take values >= 0
        c = codes[signed]
        add("fo_quantize", spec, timed(lambda: fo.fo_quantize(src_x, spec, c, scales, stream)), 5 * n + 2 * ng)
        add("fo_dequantize", spec, timed(lambda: fo.fo_dequantize(c, scales, spec, out, stream)), 5 * n + 2 * ng)
    # a library copy with dequantize's traffic (1 B read, 4 B written per
    # element): the write-heavy ceiling that kernel is measured against
    add("torch copy int8 -> fp32", "same bytes as fo_dequantize", timed(lambda: out.copy_(codes[True])), 5 * n)
    for rb in (8, 16):
        r = rhos[rb]
        nb = 4 * n + 2 * n + rb // 8 * n
        add("fo_split", f"rho{rb}", timed(lambda: fo.fo_split(x, rb, theta_bf, r, stream)), nb)
        add("fo_reconstruct", f"rho{rb}", timed(lambda: fo.fo_reconstruct(theta_bf, r, rb, out, stream)), nb)
    return {"pair_kernels": rows, "n": n, "peak_gbs": peak, "peak_source": src, "reps": reps,
            "timing": "CUDA events on the launching stream; inputs far larger than L2"}


# ------------------------------------------------------------ main
def max_over_ranks(ms: float, device) -> float:
    """The slowest rank's step time: every rank must have finished a step for
    the job to have finished it (a no-op outside torch.distributed)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return ms
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(params_per_rank: int, world_size: int, ms: float) -> float:
    """Parameters the whole job steps per second: each rank steps its own list
    (weak scaling), the job takes as long as its slowest rank."""
    return world_size * params_per_rank / (ms * 1e-3)


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--workload", default=W.LLAMA3_8B.name, choices=sorted(WORKLOADS) + [SINGLE],
                    help="tensor list: llama-3-8b (int8 rho, the headline) or llama-1.1b (int16 rho); "
                         f"{SINGLE}: the single 65,553-parameter tensor (latency-bound, parity-test size)")
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=8)
    ap.add_argument("--cpu-sample", type=int, default=436_224_000,
                    help="parameters of the CPU-oracle sample (default: two decoder layers, ~10 s of work)")
    ap.add_argument("--cpu-steps", type=int, default=20)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--layers", type=int, default=None,
                    help="profiling only: restrict to the first N decoder layers' tensors")
    ap.add_argument("--host-link", action="store_true",
                    help="only measure pinned host <-> device copy bandwidth and print it as JSON")
    ap.add_argument("--per-tensor", action="store_true",
                    help="time the step as gradient release launches it: one single-tensor launch per tensor")
    ap.add_argument("--pairs", action="store_true",
                    help="time the standalone kernels (fo_quantize / fo_dequantize / fo_split / "
                         "fo_reconstruct) on 2^30 elements and print their achieved GB/s")
    ap.add_argument("--optimizer", default="adamw", choices=["adamw", "sgd"],
                    help="sgd: time FlashSGD (fo_sgd_step, momentum = beta1) in --format "
                         "(default bf16_rho8:companded)")
    ap.add_argument("--format", default=None,
                    help="PARAM:STATES, e.g. bf16:linear or f32:f32 -- time fo_adamw_step_general in an "
                         "ablation format (parameter: bf16_rho8, bf16_rho16, bf16, f32; states: companded, "
                         "linear, f32) instead of the fast step")
    args = ap.parse_args()
    if args.workload == SINGLE:
        if args.impl != "gb300":
            raise SystemExit("the single-tensor workload has no reference arm")
        import quantized_state_optimizer_gb300 as fo
        fo.lib()
        torch.cuda.set_device(0)
        print(json.dumps(single_tensor_line(args.steps, args.warmup, torch.device("cuda", 0))), flush=True)
        return
    use_workload(args.workload)
    ws, rank, local = dist_env()
    numels = [s.numel for s in W.llama_tensor_list(MODEL)]

    if args.impl == "reference":
        if rank != 0:
            return
        # each step: the oracle over a bounded 8M-parameter sample of the workload
        cores = host_cores()
        pieces = oracle_sample(8 << 20)
        n = sum(p[0].numel for p in pieces)
        run_oracle_steps(pieces, args.warmup, cores)
        sec = run_oracle_steps(pieces, args.steps, cores, t0=args.warmup + 1)
        v = n * args.steps / sec
        line = {"metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": 1e3 * sec / args.steps, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
                "impl": "reference", "config": workload_config(numels),
                "cpu_baseline": {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle",
                                 "sample": f"{n:,} params of layer 0 per step (group-aligned 1M pieces), "
                                           f"one thread per piece on {cores} host cores"},
                "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
                "gpu_launches": 0}
        print(json.dumps(line), flush=True)
        return

    if args.host_link:
        print(json.dumps({"host_link": host_link()}), flush=True)
        return
    if args.pairs:
        print(json.dumps(pair_kernels()), flush=True)
        return

    dist_on = ws > 1
    if dist_on:
        torch.distributed.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    import quantized_state_optimizer_gb300 as fo
    fo.lib()  # fail loudly if the CUDA library is missing

    if args.optimizer == "sgd" and args.format is None:
        args.format = "bf16_rho8:companded"
    st, numels = build_state(device, args.layers, args.format, args.optimizer)
    slabs = grad_sets(st, args.layers, device)
    stream = torch.cuda.Stream(device=device)
    stepper = BenchSteps(st, slabs, per_tensor=args.per_tensor)
    launches_per_step = stepper.launches_per_step
    with ClockSampler(local) as clk:
        total_ms, per = time_steps(stepper, args.steps, args.warmup, stream, dist_on)
    ms = max_over_ranks(total_ms / args.steps, device)
    n = sum(numels)
    value = job_throughput(n, ws, ms)
    bytes_step = (algorithmic_bytes(numels) if args.format is None
                  else int(round(general_bytes_per_param(*args.format.split(":"), args.optimizer) * sum(numels))))
    kernel_ms = statistics.mean(per)
    peak, peak_kind = load_peak()
    achieved = bytes_step / (kernel_ms * 1e-3) / 1e9
    try:
        e2e = (time_e2e(st, numels, args.e2e_steps, stream, slabs)
               if args.e2e_steps > 0 and args.format is None and not args.per_tensor else None)
        if e2e is not None:
            # the link's own ceiling on this machine, for reading the e2e number
            link = host_link(gib=2)
            moved = e2e["h2d_bytes_per_step"] + e2e["d2h_bytes_per_step"]
            e2e["link_both_directions_gbs"] = link["both_directions_gbs"]
            e2e["link_floor_ms"] = moved / 1e9 / link["both_directions_gbs"] * 1e3
    except RuntimeError as exc:  # e.g. pinned host memory unavailable: keep the device number
        e2e = {"value": None, "unit": UNIT, "error": str(exc).splitlines()[0][:200]}
    footprint = st.bytes_allocated() if hasattr(st, "bytes_allocated") else None
    del st, stepper, slabs
    torch.cuda.empty_cache()

    if rank != 0:
        if dist_on:
            torch.distributed.destroy_process_group()
        return
    cpu = None
    if not args.no_cpu_baseline:
        cpu = cpu_baseline(args.cpu_sample, args.cpu_steps)
    cfg = workload_config(numels)
    if args.layers is not None:
        cfg["workload"] = f"PROFILING SUBSET (first {args.layers} layers) of " + cfg["workload"]
    if args.format is not None:
        entry = "fo_sgd_step, FlashSGD, momentum 0.9" if args.optimizer == "sgd" else "fo_adamw_step_general"
        cfg["workload"] = (f"FORMAT {args.format} ({entry}, {step_kernel_name(args.format, args.optimizer)}) of the "
                           f"{MODEL.name} list: {len(numels)} tensors, {sum(numels):,} params, bf16 grads")
    if args.per_tensor:
        cfg["workload"] = (f"PER-TENSOR LAUNCHES (the gradient-release step: {len(numels)} single-tensor "
                           f"fo_adamw_step launches per step, back to back) of " + cfg["workload"])
    if footprint is not None:
        # the state's HBM footprint between steps (grads included) against the
        # paper's storage accounting for this format
        from quantized_state_optimizer_gb300.accounting import storage_bytes_per_param
        cfg["state_bytes_per_param"] = footprint / n
        cfg["state_bytes_per_param_accounted"] = storage_bytes_per_param(
            "bf16_rho8" if RHO_BITS == 8 else "bf16_rho16", "companded")["total"]
    cfg["bytes_per_step"] = bytes_step
    cfg["bytes_per_param"] = bytes_step / n
    cfg["hbm_gbs"] = achieved
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "ms_per_step_median": statistics.median(per),
        "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic", "config": cfg,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_source": f"{peak_kind} copy bandwidth",
                     "frac_of_nominal_8000_gbs": achieved / 8000.0,
                     "kernel": step_kernel_name(args.format, args.optimizer),
                     "kernel_ms": kernel_ms, "bytes_per_launch": bytes_step,
                     "traffic": (captured_traffic(n, step_kernel_name(args.format, args.optimizer), args.format)
                                 if args.layers is None and not args.per_tensor else None)},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": args.steps * launches_per_step,
        "clocks": clk.summary(),
    }
    print(json.dumps(line), flush=True)
    if dist_on:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
