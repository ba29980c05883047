"""FlashAdamW state containers and a ``torch.optim.Optimizer`` front end.

``FlashAdamWState`` holds the optimizer state of a list of tensors in a few
flat device slabs (one per buffer kind), each tensor at a 16-byte-aligned
offset, and drives ``fo_adamw_step`` over the whole list in one call.

``FlashAdamW`` is the drop-in optimizer for bf16 ``torch.nn.Parameter`` s,
following ``FlashAdamWSim`` of the page "code/flashsim/flash_adamw_sim.py":
lazily initialised state (quantized zeros, theta split on first use), the
step count incremented before the update, parameters without a gradient
skipped.  All arithmetic runs in libfo.so.
"""

from __future__ import annotations

import torch

from . import FoTensor, FoTensorGeneral, fo_adamw_step, fo_sgd_step, fo_split, n_groups

_ALIGN_BYTES = 16


def _align(n_elems: int, elem_bytes: int) -> int:
    per = _ALIGN_BYTES // elem_bytes if elem_bytes < _ALIGN_BYTES else 1
    return (n_elems + per - 1) // per * per


class FlashAdamWState:
    """Flat device buffers for the FlashAdamW state of ``numels`` tensors.

    Per tensor: theta' (bf16), rho (int8 or int16), m codes (int8), m scales
    (fp16), v codes (uint8), v scales (fp16), and optionally a grad buffer
    (fp32 or bf16).  All start at zero: zero codes and scales are the
    quantized zero state.
    """

    def __init__(self, numels, rho_bits: int = 8, grad_dtype=torch.bfloat16, device="cuda",
                 with_grads: bool = True):
        if rho_bits not in (8, 16):
            raise ValueError("rho_bits must be 8 or 16")
        self.numels = [int(n) for n in numels]
        self.rho_bits = rho_bits
        self.grad_dtype = grad_dtype
        self.device = torch.device(device)
        rho_dt = torch.int8 if rho_bits == 8 else torch.int16
        self._off, self._goff = [], []
        o = go = 0
        for n in self.numels:
            self._off.append(o)
            self._goff.append(go)
            o += _align(n, 1) if n else 0       # 16 elements: keeps every slab 16-byte aligned
            go += _align(n_groups(n), 2) if n else 0
        total, gtotal = max(o, 16), max(go, 8)
        dev = self.device
        self.param = torch.zeros(total, dtype=torch.bfloat16, device=dev)
        self.rho = torch.zeros(total, dtype=rho_dt, device=dev)
        self.m_codes = torch.zeros(total, dtype=torch.int8, device=dev)
        self.v_codes = torch.zeros(total, dtype=torch.uint8, device=dev)
        self.m_scales = torch.zeros(gtotal, dtype=torch.float16, device=dev)
        self.v_scales = torch.zeros(gtotal, dtype=torch.float16, device=dev)
        self.grad = torch.zeros(total, dtype=grad_dtype, device=dev) if with_grads else None
        self._fo_array = None

    # ------------------------------------------------------------ views
    def __len__(self) -> int:
        return len(self.numels)

    def _v(self, slab, i, n):
        return slab[self._off[i]: self._off[i] + n]

    def view(self, i: int) -> dict[str, torch.Tensor]:
        n = self.numels[i]
        g = n_groups(n)
        go = self._goff[i]
        d = {
            "param": self._v(self.param, i, n), "rho": self._v(self.rho, i, n),
            "m_codes": self._v(self.m_codes, i, n), "v_codes": self._v(self.v_codes, i, n),
            "m_scales": self.m_scales[go: go + g], "v_scales": self.v_scales[go: go + g],
        }
        if self.grad is not None:
            d["grad"] = self._v(self.grad, i, n)
        return d

    def grad_view(self, i: int) -> torch.Tensor:
        return self._v(self.grad, i, self.numels[i])

    def total_numel(self) -> int:
        return sum(self.numels)

    def bytes_allocated(self) -> int:
        """Device bytes of every slab (the state's HBM footprint, padding included)."""
        slabs = [self.param, self.rho, self.m_codes, self.v_codes, self.m_scales, self.v_scales]
        if self.grad is not None:
            slabs.append(self.grad)
        return sum(t.numel() * t.element_size() for t in slabs)

    # ------------------------------------------------------------ set-up
    def init_theta(self, i: int, theta: torch.Tensor, stream=None) -> None:
        """Split an fp32 master weight into this tensor's theta' and rho."""
        v = self.view(i)
        fo_split(theta.reshape(-1).contiguous(), self.rho_bits, v["param"], v["rho"], stream)

    def fo_tensors(self, grads=None):
        """ctypes array of ``fo_tensor`` for all tensors (cached for the slab grads)."""
        if grads is None and self._fo_array is not None:
            return self._fo_array
        arr = (FoTensor * max(len(self.numels), 1))()
        for i, n in enumerate(self.numels):
            v = self.view(i)
            g = v["grad"] if grads is None else grads[i]
            arr[i] = FoTensor(v["param"].data_ptr(), v["rho"].data_ptr(), g.data_ptr(),
                              v["m_codes"].data_ptr(), v["m_scales"].data_ptr(),
                              v["v_codes"].data_ptr(), v["v_scales"].data_ptr(), n)
        if grads is None:
            self._fo_array = arr
        return arr

    def step(self, step: int, lr: float, beta1: float, beta2: float, eps: float,
             weight_decay: float, grads=None, stream=None) -> None:
        """One fused FlashAdamW step over every tensor (one kernel launch)."""
        arr = self.fo_tensors(grads)
        gdt = self.grad_dtype if grads is None else grads[0].dtype
        fo_adamw_step(arr, gdt, lr, beta1, beta2, eps, weight_decay, step, self.rho_bits, stream)

    def _chunks(self, n_chunks: int):
        """Contiguous groups of tensors with about equal element counts:
        (first tensor, end tensor, slab start, slab end) each."""
        key = ("chunks", n_chunks)
        if getattr(self, "_chunk_key", None) == key:
            return self._chunk_list
        total = max(self.total_numel(), 1)
        out, first, acc = [], 0, 0
        for i, n in enumerate(self.numels):
            acc += n
            if acc * n_chunks >= total * (len(out) + 1) or i == len(self.numels) - 1:
                end = i + 1
                lo = self._off[first]
                hi = self._off[end] if end < len(self.numels) else self.param.numel()
                arr = (FoTensor * (end - first))(*[self.fo_tensors()[j] for j in range(first, end)])
                out.append((first, end, lo, hi, arr))
                first = end
        self._chunk_key, self._chunk_list = key, out
        return out

    def step_from_host(self, step: int, lr: float, beta1: float, beta2: float, eps: float,
                       weight_decay: float, host_grad: torch.Tensor, host_param: torch.Tensor,
                       n_chunks: int = 8, stream=None) -> None:
        """One step fed from host memory: upload the gradients from ``host_grad``
        (pinned, laid out like the grad slab), step, and download the new theta'
        into ``host_param`` (pinned, laid out like the param slab).

        The list is cut into ``n_chunks`` groups of tensors.  Chunk c's upload,
        step launch and download run on three streams chained by events, so the
        copies of one chunk overlap the step of another and the two copy
        directions overlap each other.  Everything is ordered after the work
        already on ``stream`` (default: the current stream), and ``stream``
        waits for the last download, so a later step or a synchronize on it
        sees the finished parameters."""
        if self.grad is None:
            raise RuntimeError("step_from_host needs the grad slab (with_grads=True)")
        if host_grad.numel() != self.grad.numel() or host_param.numel() != self.param.numel():
            raise ValueError("host buffers must match the grad and param slabs")
        compute = stream if stream is not None else torch.cuda.current_stream(self.device)
        if not hasattr(self, "_copy_streams"):
            self._copy_streams = (torch.cuda.Stream(self.device), torch.cuda.Stream(self.device))
        up, down = self._copy_streams
        up.wait_stream(compute)  # the previous step no longer reads the grad slab
        down.wait_stream(compute)
        for first, end, lo, hi, arr in self._chunks(n_chunks):
            with torch.cuda.stream(up):
                self.grad[lo:hi].copy_(host_grad[lo:hi], non_blocking=True)
                uploaded = torch.cuda.Event()
                uploaded.record(up)
            compute.wait_event(uploaded)
            fo_adamw_step(arr, self.grad_dtype, lr, beta1, beta2, eps, weight_decay, step, self.rho_bits,
                          compute)
            stepped = torch.cuda.Event()
            stepped.record(compute)
            down.wait_event(stepped)
            with torch.cuda.stream(down):
                host_param[lo:hi].copy_(self.param[lo:hi], non_blocking=True)
        compute.wait_stream(down)

    def state_dict(self) -> dict[str, torch.Tensor]:
        """Host copies of every state slab (checkpoint)."""
        return {k: getattr(self, k).cpu() for k in
                ("param", "rho", "m_codes", "m_scales", "v_codes", "v_scales")}

    def load_state_dict(self, sd: dict[str, torch.Tensor]) -> None:
        for k, t in sd.items():
            getattr(self, k).copy_(t)


class FlashAdamW(torch.optim.Optimizer):
    """AdamW with 8-bit group-quantized m and v and a bf16 + rho master weight.

    Parameters must be bf16 CUDA tensors; their fp32 master weights live as
    (theta' = the parameter itself, rho).  ``master_weight_bits`` = 24 (int8
    rho) or 32 (int16 rho).  Gradients may be bf16 or fp32 (one dtype per
    step call).  All parameters of all groups that have a gradient are updated
    by one launch per param group.

    ``gradient_release=True`` steps each parameter inside backward instead:
    a post-accumulate-grad hook launches the single-tensor step as soon as
    the parameter's gradient is complete and then frees the gradient, so no
    gradient outlives its own update (the ``gradient_release`` accounting of
    ``bytes_per_param`` on the page "code/flashsim/flash_adamw_sim.py").
    Parameters of fewer than ``release_bucket_numel`` elements (norm weights,
    say) are gathered instead: their group's bucket is stepped in one launch
    once every such parameter of the group has its gradient, or at
    ``step()`` for any left over, so those few small gradients live until
    their bucket's update.  ``step()`` does nothing else for released
    parameters.  The result equals a normal step on the same gradients bit
    for bit: every tensor's update is independent of the others.
    """

    def __init__(self, params, lr=1e-3, betas=(0.9, 0.999), eps=1e-8, weight_decay=0.0,
                 master_weight_bits: int = 24, gradient_release: bool = False,
                 release_bucket_numel: int = 1 << 20):
        if master_weight_bits not in (24, 32):
            raise ValueError("master_weight_bits must be 24 or 32")
        defaults = dict(lr=lr, betas=betas, eps=eps, weight_decay=weight_decay)
        super().__init__(params, defaults)
        self.rho_bits = 8 if master_weight_bits == 24 else 16
        self.gradient_release = gradient_release
        self.release_bucket_numel = int(release_bucket_numel)
        self._hooks = []
        self._args = {}     # parameter -> its one-entry fo_tensor array (state pointers fixed)
        self._pending = {}  # group index -> small parameters whose gradients are complete
        self._n_small = {}  # group index -> number of small parameters in the group
        if gradient_release:
            for gi, group in enumerate(self.param_groups):
                small = [p for p in group["params"] if p.numel() < self.release_bucket_numel]
                self._n_small[gi] = len(small)
                for p in group["params"]:
                    self._hooks.append(p.register_post_accumulate_grad_hook(self._release_hook(gi, group)))

    def _release_hook(self, gi: int, group):
        def hook(p: torch.Tensor) -> None:
            if p.numel() < self.release_bucket_numel:
                pend = self._pending.setdefault(gi, [])
                pend.append(p)
                if len(pend) == self._n_small[gi]:
                    self._flush(gi)
                return
            with torch.no_grad():
                self._step_one(group, p)
            p.grad = None
        return hook

    def _flush(self, gi: int) -> None:
        """Step a group's gathered small parameters in one launch and free their gradients."""
        pend = self._pending.pop(gi, [])
        if pend:
            with torch.no_grad():
                self._step_params(self.param_groups[gi], pend)
            for p in pend:
                p.grad = None

    def _step_one(self, group, p: torch.Tensor) -> None:
        """The single-tensor step of a released parameter through its cached argument array."""
        st = self.state[p]
        if len(st) == 0:
            st = self._init_state(p)
        arr = self._args.get(p)
        if arr is None:
            arr = (FoTensor * 1)(FoTensor(p.data_ptr(), st["rho"].data_ptr(), 0, st["m_codes"].data_ptr(),
                                          st["m_scales"].data_ptr(), st["v_codes"].data_ptr(),
                                          st["v_scales"].data_ptr(), p.numel()))
            self._args[p] = arr
        st["step"] += 1
        g = p.grad if p.grad.is_contiguous() else p.grad.contiguous()
        arr[0].grad = g.data_ptr()
        beta1, beta2 = group["betas"]
        fo_adamw_step(arr, g.dtype, group["lr"], beta1, beta2, group["eps"], group["weight_decay"], st["step"],
                      self.rho_bits)

    def load_state_dict(self, state_dict) -> None:
        super().load_state_dict(state_dict)
        self._args = {}  # the state buffers were replaced

    def remove_hooks(self) -> None:
        """Detach the gradient-release hooks (the optimizer then steps in ``step()``)."""
        for gi in list(self._pending):
            self._flush(gi)
        for h in self._hooks:
            h.remove()
        self._hooks = []
        self.gradient_release = False

    def _init_state(self, p: torch.Tensor) -> dict:
        if p.dtype != torch.bfloat16 or not p.is_cuda or not p.is_contiguous():
            raise TypeError("FlashAdamW parameters must be contiguous bf16 CUDA tensors")
        n = p.numel()
        dev = p.device
        st = self.state[p]
        st["step"] = 0
        st["rho"] = torch.zeros(n, dtype=torch.int8 if self.rho_bits == 8 else torch.int16, device=dev)
        st["m_codes"] = torch.zeros(n, dtype=torch.int8, device=dev)
        st["m_scales"] = torch.zeros(n_groups(n), dtype=torch.float16, device=dev)
        st["v_codes"] = torch.zeros(n, dtype=torch.uint8, device=dev)
        st["v_scales"] = torch.zeros(n_groups(n), dtype=torch.float16, device=dev)
        # the parameter is already bf16: its master starts as the parameter itself (rho = 0)
        return st

    @torch.no_grad()
    def step(self, closure=None):
        loss = None
        if closure is not None:
            with torch.enable_grad():
                loss = closure()
        if not self.gradient_release:
            for group in self.param_groups:
                self._step_params(group, group["params"])
        else:
            for gi in list(self._pending):  # small parameters whose bucket did not fill
                self._flush(gi)
        return loss

    def _step_params(self, group, params) -> None:
        """One launch per (step count, grad dtype) over the parameters that have a gradient."""
        beta1, beta2 = group["betas"]
        by_key: dict[tuple[int, torch.dtype], list] = {}
        for p in params:
            if p.grad is None:
                continue
            st = self.state[p]
            if len(st) == 0:
                st = self._init_state(p)
            st["step"] += 1
            g = p.grad
            if not g.is_contiguous():
                g = g.contiguous()
            ft = FoTensor(p.data_ptr(), st["rho"].data_ptr(), g.data_ptr(), st["m_codes"].data_ptr(),
                          st["m_scales"].data_ptr(), st["v_codes"].data_ptr(),
                          st["v_scales"].data_ptr(), p.numel())
            by_key.setdefault((st["step"], g.dtype), []).append((ft, g))
        for (t, gdt), items in by_key.items():
            fo_adamw_step([ft for ft, _ in items], gdt, group["lr"], beta1, beta2, group["eps"],
                          group["weight_decay"], t, self.rho_bits)


class FlashSGD(torch.optim.Optimizer):
    """SGD with momentum on bf16 parameters with a split master weight and an
    8-bit group-quantized momentum buffer (``fo_sgd_step``; the update rule is
    the reading stated in include/fo.h).  ``master_weight_bits`` = 24 (int8 rho)
    or 32 (int16 rho).  One launch per (param group, grad dtype)."""

    def __init__(self, params, lr=1e-2, momentum=0.9, weight_decay=0.0, master_weight_bits: int = 24):
        if master_weight_bits not in (24, 32):
            raise ValueError("master_weight_bits must be 24 or 32")
        super().__init__(params, dict(lr=lr, momentum=momentum, weight_decay=weight_decay))
        self.rho_bits = 8 if master_weight_bits == 24 else 16

    @torch.no_grad()
    def step(self, closure=None):
        loss = None
        if closure is not None:
            with torch.enable_grad():
                loss = closure()
        pf = "bf16_rho8" if self.rho_bits == 8 else "bf16_rho16"
        for group in self.param_groups:
            by_dtype: dict[torch.dtype, list] = {}
            for p in group["params"]:
                if p.grad is None:
                    continue
                if p.dtype != torch.bfloat16 or not p.is_cuda or not p.is_contiguous():
                    raise TypeError("FlashSGD parameters must be contiguous bf16 CUDA tensors")
                st = self.state[p]
                if len(st) == 0:
                    n = p.numel()
                    st["rho"] = torch.zeros(n, dtype=torch.int8 if self.rho_bits == 8 else torch.int16,
                                            device=p.device)
                    st["m_codes"] = torch.zeros(n, dtype=torch.int8, device=p.device)
                    st["m_scales"] = torch.zeros(n_groups(n), dtype=torch.float16, device=p.device)
                g = p.grad if p.grad.is_contiguous() else p.grad.contiguous()
                ft = FoTensorGeneral(p.data_ptr(), st["rho"].data_ptr(), g.data_ptr(), st["m_codes"].data_ptr(),
                                     st["m_scales"].data_ptr(), None, None, p.numel())
                by_dtype.setdefault(g.dtype, []).append((ft, g))
            for gdt, items in by_dtype.items():
                fo_sgd_step([ft for ft, _ in items], pf, "companded", gdt, group["lr"], group["momentum"],
                            group["weight_decay"])
        return loss
