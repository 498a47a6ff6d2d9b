"""Caller-side plumbing around the C ABI: torch allocates the flat buffers and
owns the stream; every step of the path runs in the library's kernels.

``FlatStep`` plans the FlatParameter layout, allocates master / m / v (fp32)
and the bf16 parameter buffer of ``padded_numel`` elements on the device,
builds the master with ``zero_make_master`` and then drives the protocol:
``reduce_grads`` -> ``step`` -> ``gather_weights`` -> ``post_step``.

With ``offload=True`` (ZeRO-Offload) master / m / v are host tensors instead,
the context comes from ``zero_make_master_offload`` and ``step`` runs
``zero_offload_step``: the reduced gradient goes down to the host chunk by
chunk, the library's multi-threaded CPU Adam updates the host state and the
bf16 parameters come back up, on a second (copy) stream.
"""

from __future__ import annotations

from typing import List, Optional, Sequence

import torch

from . import binding as B


class FlatStep:
    def __init__(self, param_numel: Sequence[int], param_unit: Sequence[int], *, stage: int, n_ranks: int,
                 grad_dtype: str = "bf16", lr: float = 1e-3, beta1: float = 0.9, beta2: float = 0.999,
                 eps: float = 1e-8, weight_decay: float = 0.0, adamw: bool = False,
                 init_params: Sequence[torch.Tensor] = (), device: str | torch.device = "cuda",
                 guard: int = 0, guard_value: float = float("nan"), offload: bool = False,
                 offload_chunk: int = 1 << 23, offload_threads: int = 0):
        self.param_numel = [int(x) for x in param_numel]
        self.param_unit = [int(x) for x in param_unit]
        self.stage, self.n_ranks, self.grad_dtype = stage, n_ranks, grad_dtype
        self.cfg = B.make_config(stage, n_ranks, grad_dtype, lr, beta1, beta2, eps, weight_decay, adamw)
        self.device = torch.device(device)
        if self.device.type == "cuda" and self.device.index is None:
            self.device = torch.device("cuda", torch.cuda.current_device())
        plan = B.zero_plan(self.cfg, self.param_numel, self.param_unit)
        try:
            self.padded, self.numel = B.zero_padded_numel(plan)
            self.n_units = B.zero_num_units(plan)
        finally:
            B.zero_destroy(plan)
        # Optional guard regions around every buffer (canary checks in tests);
        # a multiple of 8 elements keeps the interior 16-byte aligned.
        if guard < 0 or guard % 8:
            raise ValueError("guard must be a non-negative multiple of 8 elements")
        self.guard = guard
        n = self.padded + 2 * guard

        def alloc(dtype, device):
            t = torch.empty(max(n, 1), dtype=dtype, device=device)
            t.fill_(guard_value)
            return t

        self.offload = bool(offload)
        state_device = torch.device("cpu") if self.offload else self.device
        self._master, self._m, self._v = (alloc(torch.float32, state_device) for _ in range(3))
        self._p16 = alloc(torch.bfloat16, self.device)
        if len(init_params) != len(self.param_numel):
            raise ValueError("need one fp32 init tensor per parameter")
        self._init = [p.contiguous() for p in init_params]
        for p, k in zip(self._init, self.param_numel):
            if p.dtype != torch.float32 or p.numel() != k:
                raise ValueError("init params must be fp32 tensors of the declared sizes")
        make = B.zero_make_master_offload if self.offload else B.zero_make_master
        self.ctx = make(self.cfg, self.param_numel, self.param_unit, [p.data_ptr() for p in self._init],
                        self._ptr(self._master), self._ptr(self._m), self._ptr(self._v),
                        self._ptr(self._p16), self.stream_handle())
        if self.offload:
            self.offload_chunk, self.offload_threads = int(offload_chunk), int(offload_threads)
            hb, db = B.zero_offload_workspace_bytes(self.ctx, self.offload_chunk)
            self._host_ws = torch.empty(hb, dtype=torch.uint8, pin_memory=True)
            self._dev_ws = torch.empty(db, dtype=torch.uint8, device=self.device)
            self._copy_stream = torch.cuda.Stream(self.device)
        # padded length of every unit, for the registration length checks
        self._unit_padded = [B.zero_layout(self.ctx, i)[1] for i in range(self.n_units)]
        # make_master reads the init params on the stream; once it has run they
        # may be released.
        torch.cuda.current_stream(self.device).synchronize()
        self._init = []
        self._registered: List[List[torch.Tensor]] = []

    # -- buffers ---------------------------------------------------------------
    def _ptr(self, t: torch.Tensor) -> int:
        return t.data_ptr() + self.guard * t.element_size()

    def _view(self, t):
        return t[self.guard:self.guard + self.padded]

    @property
    def master(self):
        return self._view(self._master)

    @property
    def exp_avg(self):
        return self._view(self._m)

    @property
    def exp_avg_sq(self):
        return self._view(self._v)

    @property
    def param16(self):
        return self._view(self._p16)

    def guards(self):
        """The guard regions of every buffer (must keep their fill value)."""
        g = self.guard
        out = []
        for t in (self._master, self._m, self._v, self._p16):
            out.append(t[:g])
            out.append(t[g + self.padded:])
        return out

    def layout(self, unit: int):
        return B.zero_layout(self.ctx, unit)

    def param_offset(self, p: int) -> int:
        return B.zero_param_offset(self.ctx, p)

    @staticmethod
    def stream_handle(stream: Optional[torch.cuda.Stream] = None) -> int:
        s = stream if stream is not None else torch.cuda.current_stream()
        return int(s.cuda_stream)

    def grad_dtype_torch(self):
        return torch.bfloat16 if self.grad_dtype == "bf16" else torch.float32

    # -- protocol ----------------------------------------------------------------
    def _need(self, unit: int) -> int:
        """Elements each replica buffer of `unit` (-1: all units) must hold:
        the padded length the kernels read, pads included."""
        if unit < 0:
            return self.padded
        if unit >= self.n_units:
            return 0  # the library reports the bad unit
        return self._unit_padded[unit]

    def reduce_grads(self, unit: int, replica_grads: Sequence[torch.Tensor], stream=None) -> None:
        want = self.grad_dtype_torch()
        need = self._need(unit)
        for g in replica_grads:
            if g.dtype != want or not g.is_contiguous() or g.device != self.device:
                raise ValueError("replica grads must be contiguous device tensors of the configured dtype")
            if g.numel() < need:
                raise ValueError(f"replica grads must hold the padded {need} elements (pads included), "
                                 f"got {g.numel()}")
        B.zero_reduce_grads(self.ctx, unit, [g.data_ptr() for g in replica_grads], self.stream_handle(stream))
        self._registered.append(list(replica_grads))  # keep alive until post_step

    def clip_grad_norm(self, max_norm: float, keep_reduced: bool = False, stream=None) -> None:
        """Global-norm clipping of the registered gradients for the next step
        (the workspace is allocated once, by torch, and reused).  keep_reduced
        lets the next step read the kept reduced gradient instead of the N
        replicas (more workspace, fewer bytes moved for N > 4)."""
        flags = B.ZERO_CLIP_KEEP_REDUCED if keep_reduced else 0
        need = B.zero_clip_workspace_bytes_ex(self.ctx, flags)
        if getattr(self, "_clip_ws", None) is None or self._clip_ws.numel() < need:
            self._clip_ws = torch.empty(need, dtype=torch.uint8, device=self.device)
        B.zero_clip_grad_norm_ex(self.ctx, max_norm, flags, self._clip_ws.data_ptr(), self._clip_ws.numel(),
                                 self.stream_handle(stream))

    def grad_norm(self, stream=None) -> float:
        """Norm of the last clip (synchronizes the stream)."""
        return B.zero_grad_norm(self.ctx, self.stream_handle(stream))

    def accumulate_grads(self, unit: int, micro_grads: Sequence[torch.Tensor], accumulators: Sequence[torch.Tensor],
                         first: bool, stream=None) -> None:
        """fp32 accumulation of one micro-step's bf16 replica gradients."""
        need = self._need(unit)
        for g in micro_grads:
            if g.dtype != torch.bfloat16 or not g.is_contiguous() or g.device != self.device:
                raise ValueError("micro gradients must be contiguous bf16 device tensors")
            if g.numel() < need:
                raise ValueError(f"micro gradients must hold the padded {need} elements, got {g.numel()}")
        for a in accumulators:
            if a.dtype != torch.float32 or not a.is_contiguous() or a.device != self.device:
                raise ValueError("accumulators must be contiguous fp32 device tensors")
            if a.numel() < need:
                raise ValueError(f"accumulators must hold the padded {need} elements, got {a.numel()}")
        B.zero_accumulate_grads(self.ctx, unit, [g.data_ptr() for g in micro_grads],
                                [a.data_ptr() for a in accumulators], first, self.stream_handle(stream))

    def step(self, stream=None) -> None:
        if self.offload:
            B.zero_offload_step(self.ctx, self.offload_chunk, self._host_ws.data_ptr(), self._host_ws.numel(),
                                self._dev_ws.data_ptr(), self._dev_ws.numel(), self.offload_threads,
                                self.stream_handle(stream), self.stream_handle(self._copy_stream))
        else:
            B.zero_step(self.ctx, self.stream_handle(stream))

    def gather_weights(self, unit: int, out: Optional[torch.Tensor], stream=None) -> None:
        """ZeRO-3: copy unit `unit` (-1: every unit) of the bf16 parameters,
        pads included, into `out`; a no-op for stages 0-2 (out may be None)."""
        if out is not None and self.stage == 3:
            need = self._need(unit)
            if out.dtype != torch.bfloat16 or not out.is_contiguous() or out.device != self.device:
                raise ValueError("the gather buffer must be a contiguous bf16 device tensor")
            if out.numel() < need:
                raise ValueError(f"the gather buffer must hold the padded {need} elements, got {out.numel()}")
        B.zero_gather_weights(self.ctx, unit, out.data_ptr() if out is not None else 0, self.stream_handle(stream))

    def gather_units(self, first_unit: int, outs: Sequence[Optional[torch.Tensor]], stream=None) -> None:
        """ZeRO-3 prefetch: units first_unit .. first_unit + len(outs) - 1
        into `outs` (one bf16 device tensor per unit, None for an empty unit)
        with one kernel per 32 units; a no-op for stages 0-2."""
        if self.stage == 3:
            for k, out in enumerate(outs):
                need = self._need(first_unit + k) if 0 <= first_unit + k < self.n_units else 0
                if out is None:
                    continue
                if out.dtype != torch.bfloat16 or not out.is_contiguous() or out.device != self.device:
                    raise ValueError("a gather buffer must be a contiguous bf16 device tensor")
                if out.numel() < need:
                    raise ValueError(f"the gather buffer of unit {first_unit + k} must hold the padded {need} "
                                     f"elements, got {out.numel()}")
        B.zero_gather_units(self.ctx, first_unit, [o.data_ptr() if o is not None else 0 for o in outs],
                            self.stream_handle(stream))

    def post_step(self, stream=None) -> None:
        B.zero_post_step(self.ctx, self.stream_handle(stream))
        self._registered.clear()

    def export_state(self, stream=None):
        """Layout-free checkpoint: (master, exp_avg, exp_avg_sq) fp32 device
        tensors of the real elements in parameter order, and the step count."""
        out = [torch.empty(max(self.numel, 1), dtype=torch.float32, device=self.device) for _ in range(3)]
        t = B.zero_export_state(self.ctx, *[o.data_ptr() for o in out], self.stream_handle(stream))
        return [o[:self.numel] for o in out], t

    def import_state(self, master, exp_avg, exp_avg_sq, t: int, stream=None) -> None:
        for x in (master, exp_avg, exp_avg_sq):
            if x.dtype != torch.float32 or not x.is_contiguous() or x.numel() != self.numel:
                raise ValueError("state tensors must be contiguous fp32 of numel_total elements")
        B.zero_import_state(self.ctx, master.data_ptr(), exp_avg.data_ptr(), exp_avg_sq.data_ptr(), t,
                            self.stream_handle(stream))
        torch.cuda.current_stream(self.device).synchronize()

    def enable_capturable(self, max_steps: int, stream=None) -> None:
        """Capturable mode (CUDA graphs): the step count and the bias
        corrections of steps 1..max_steps live in a device workspace, so a
        captured step can be replayed.  The workspace is allocated by torch."""
        need = B.zero_capturable_workspace_bytes(self.ctx, max_steps)
        self._cap_ws = torch.empty(need, dtype=torch.uint8, device=self.device)
        B.zero_enable_capturable(self.ctx, self._cap_ws.data_ptr(), need, max_steps, self.stream_handle(stream))

    def disable_capturable(self, stream=None) -> None:
        B.zero_disable_capturable(self.ctx, self.stream_handle(stream))
        self._cap_ws = None

    def count_nonfinite(self, counter: Optional[torch.Tensor]) -> None:
        """Every later step adds its number of non-finite reduced gradients to
        `counter` (a one-element int64 device tensor, zeroed by the caller);
        None stops counting."""
        if counter is not None and (counter.dtype != torch.int64 or counter.device != self.device):
            raise ValueError("the counter must be an int64 tensor on the context's device")
        B.zero_count_nonfinite(self.ctx, counter.data_ptr() if counter is not None else 0)
        self._nonfinite = counter

    def kernel_timeouts(self) -> int:
        """Bounded waits of the tile-staged step kernels that gave up (process-wide count)."""
        return B.zero_kernel_timeouts(self.ctx)

    def step_count(self) -> int:
        return B.zero_step_count(self.ctx)

    def last_launches(self) -> int:
        """Kernels enqueued by the last step / gather call."""
        return B.zero_last_launches(self.ctx)

    def close(self) -> None:
        if getattr(self, "ctx", None):
            B.zero_destroy(self.ctx)
            self.ctx = None

    def __del__(self):  # pragma: no cover
        try:
            self.close()
        except Exception:
            pass
