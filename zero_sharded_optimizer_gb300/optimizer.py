"""User-facing ZeRO optimizer over N simulated data-parallel ranks on one GPU.

Wraps the C ABI: allocates the flat state (m, v, and the fp32 master in mixed
precision) with PyTorch, keeps the step counter, and runs one fused step per
call. Gradients may be CUDA tensors, or host tensors (ideally pinned): those go
through zero_step_from_host, which copies them into device staging buffers
chunk by chunk on a copy stream while earlier chunks are being stepped, and can
copy the updated parameters back to a host buffer on a second copy stream.

Checkpoint/resume: ``state_dict()`` / ``load_state_dict()`` copy the flat
state and the step counter; continuing from a loaded state is bit-identical
to an uninterrupted run because the step is a pure function of (state, grads).
"""

from __future__ import annotations

import torch

from . import abi

BUCKET_BYTES_25MIB = 25 * 1024 * 1024


class ZeroOptimizer:
    def __init__(self, n: int, N: int, precision: int = abi.ZERO_FP32, lr: float = 1e-3,
                 betas=(0.9, 0.999), eps: float = 1e-8, weight_decay: float = 0.0,
                 master_init: torch.Tensor | None = None, device="cuda", stream=None,
                 max_grad_norm: float = 0.0, grad_scale: float = 1.0, shard_bounds=None,
                 stage: int = 2, optimizer: str = "adamw", momentum: float = 0.0,
                 dampening: float = 0.0, nesterov: bool = False):
        """``max_grad_norm`` > 0 clips the (scaled) mean gradient to that global
        norm before every step; ``grad_scale`` multiplies the mean gradient
        (1/k when the gradient buffers hold the sum of k micro-batches);
        ``shard_bounds`` (N+1 offsets) replaces the np.array_split shards, e.g.
        ``abi.zero_tensor_shard_bounds(tensor_sizes, N)`` for whole-tensor shards.
        ``stage`` 3 leaves the all-gather out of the step: each replica keeps
        only its own shard current until ``gather`` (stages 1 and 2 run the
        same fused step; they differ only in what a rank would keep).
        ``optimizer`` "sgd" runs momentum SGD (torch.optim.SGD semantics:
        ``momentum``, ``dampening``, ``nesterov``, coupled ``weight_decay``;
        ``betas`` and ``eps`` unused) with one fp32 buffer per parameter (none
        without momentum) instead of AdamW's m and v."""
        if stage not in (1, 2, 3):
            raise ValueError("stage must be 1, 2 or 3")
        if optimizer not in ("adamw", "sgd"):
            raise ValueError("optimizer must be 'adamw' or 'sgd'")
        self.optimizer = optimizer
        self.momentum, self.dampening = float(momentum), float(dampening)
        self.nesterov = bool(nesterov)
        self.stage = int(stage)
        self.shard_bounds = None if shard_bounds is None else [int(b) for b in shard_bounds]
        self.n, self.N, self.precision = int(n), int(N), int(precision)
        self.max_grad_norm, self.grad_scale = float(max_grad_norm), float(grad_scale)
        self._norm = None
        self._norm_scratch = None
        self.lr, self.beta1, self.beta2 = float(lr), float(betas[0]), float(betas[1])
        self.eps, self.weight_decay = float(eps), float(weight_decay)
        self.device = torch.device(device)
        f32 = dict(dtype=torch.float32, device=self.device)
        sgd = optimizer == "sgd"
        self.m = None if sgd and self.momentum == 0 else torch.empty(self.n, **f32)
        self.v = None if sgd else torch.empty(self.n, **f32)
        self.master = None
        if self.precision == abi.ZERO_BF16_MIXED:
            if master_init is None:
                raise ValueError("mixed precision needs the fp32 initial weights (master_init)")
            self.master = torch.empty(self.n, **f32)
            master_init = master_init.to(self.device, torch.float32).contiguous()
        self.states = abi.zero_init_states(self.n, self.N, self.precision, self.m, self.v,
                                           self.master, master_init, stream, self.shard_bounds)
        self.t = 0
        self._staging = None

    # ------------------------------------------------------------------ step --

    def _staging_buffers(self):
        if self._staging is None:
            dt = torch.bfloat16 if self.precision == abi.ZERO_BF16_MIXED else torch.float32
            self._staging = [torch.empty(self.n, dtype=dt, device=self.device)
                             for _ in range(self.N)]
            self._h2d = torch.cuda.Stream(self.device)
            self._d2h = torch.cuda.Stream(self.device)
        return self._staging

    def step(self, params, grads, stream=None, host_params_out=None,
             chunk_bytes: int = BUCKET_BYTES_25MIB) -> int:
        """One ZeRO step; returns the new step number t.

        With host gradients the copies are pipelined with the step; with
        clipping each chunk's part of the norm is summed as soon as the chunk
        has arrived, and once all are in the chunks are stepped and copied back
        one after another. Clipping uses this optimizer's own norm buffers
        (``_norm`` receives the squared norm). When
        ``host_params_out`` (a host tensor of n elements) is given, the updated
        parameters are copied into it as well; at stage 3 each shard comes from
        its owner's replica and the replicas stay released. Synchronize
        ``stream`` (the current stream by default) before reading it.
        """
        clipping = self.max_grad_norm > 0
        owner_only = self.stage == 3
        sgd = self.optimizer == "sgd"
        norm = scratch = None
        if clipping:  # the step computes the norm into self._norm itself
            norm, scratch = self._norm_buffers()
        if all(g.is_cuda for g in grads):
            if clipping or owner_only or sgd or self.grad_scale != 1.0:
                if sgd:
                    abi.zero_step_sgd(params, grads, self.states, self.t + 1, self.lr,
                                      self.momentum, self.dampening, self.weight_decay,
                                      self.nesterov, self.grad_scale, self.max_grad_norm, norm,
                                      0, -1, stream, owner_only, norm_scratch=scratch)
                else:
                    abi.zero_step_ex(params, grads, self.states, self.t + 1, self.lr,
                                     self.beta1, self.beta2, self.eps, self.weight_decay,
                                     self.grad_scale, self.max_grad_norm, norm, 0, -1, stream,
                                     owner_only, norm_scratch=scratch)
            else:
                abi.zero_step(params, grads, self.states, self.t + 1, self.lr, self.beta1,
                              self.beta2, self.eps, self.weight_decay, stream)
            if host_params_out is not None:
                s = stream if stream is not None else torch.cuda.current_stream(self.device)
                with torch.cuda.stream(s):
                    if owner_only:  # each shard from its owner's replica (no gather)
                        for r, (lo, hi) in enumerate(self._bounds_pairs()):
                            if hi > lo:
                                host_params_out[lo:hi].copy_(params[r][lo:hi], non_blocking=True)
                    else:
                        host_params_out.copy_(params[0], non_blocking=True)
        else:
            staging = self._staging_buffers()
            nq = None if norm is None else norm.data_ptr()
            sq, count = (None, 0) if scratch is None else (scratch.data_ptr(), scratch.numel())
            if sgd:
                o = abi.SgdOpts(self.t + 1, self.lr, self.momentum, self.dampening,
                                self.weight_decay, 1 if self.nesterov else 0, self.grad_scale,
                                self.max_grad_norm, nq, 0, -1, 1 if owner_only else 0, sq, count)
                abi.zero_step_from_host_ex(params, grads, staging, self.states, sgd=o,
                                           host_params_out=host_params_out,
                                           chunk_bytes=chunk_bytes, compute=stream, h2d=self._h2d,
                                           d2h=self._d2h)
            elif clipping or owner_only or self.grad_scale != 1.0:
                o = abi.StepOpts(self.t + 1, self.lr, self.beta1, self.beta2, self.eps,
                                 self.weight_decay, self.grad_scale, self.max_grad_norm, nq,
                                 0, -1, 1 if owner_only else 0, sq, count)
                abi.zero_step_from_host_ex(params, grads, staging, self.states, adamw=o,
                                           host_params_out=host_params_out,
                                           chunk_bytes=chunk_bytes, compute=stream, h2d=self._h2d,
                                           d2h=self._d2h)
            else:
                abi.zero_step_from_host(params, grads, staging, self.states, self.t + 1, self.lr,
                                        self.beta1, self.beta2, self.eps, self.weight_decay,
                                        host_params_out, chunk_bytes, stream, self._h2d,
                                        self._d2h)
        self.t += 1
        return self.t

    def _norm_buffers(self):
        """This optimizer's own device buffers for the clipping norm: the
        squared norm and the scratch of its partial sums (never shared with
        another optimizer, so optimizers on different streams do not race)."""
        f64 = dict(dtype=torch.float64, device=self.device)
        if self._norm_scratch is None:
            count = abi.zero_grad_norm_scratch_count(self.n, self.precision)
            self._norm_scratch = torch.empty(count, **f64)
        if self._norm is None:
            self._norm = torch.empty(1, **f64)
        return self._norm, self._norm_scratch

    def _bounds_pairs(self):
        b = self.shard_bounds if self.shard_bounds is not None else \
            abi.zero_shard_bounds(self.n, self.N)
        return list(zip(b[:-1], b[1:]))

    def gather(self, params, lo: int = 0, hi: int = -1, stream=None) -> None:
        """ZeRO-3 gather: every replica receives each shard from its owner's
        replica over [lo, hi) (hi < 0: n), e.g. one layer before its forward."""
        abi.zero_gather(params, self.states, lo, hi, stream)

    def step_bucketed(self, params, grads, ready=None, side=None,
                      bucket_bytes: int = BUCKET_BYTES_25MIB, done=None,
                      timeout_ms: int = -1) -> int:
        """The step bucket by bucket on ``side``, each after its ``ready`` event."""
        if self.stage == 3 or self.optimizer != "adamw":
            raise ValueError("bucket streaming runs the stage-1/2 AdamW step (with all-gather)")
        try:
            abi.zero_step_bucketed(params, grads, self.states, self.t + 1, self.lr, self.beta1,
                                   self.beta2, self.eps, self.weight_decay, bucket_bytes, ready,
                                   side, done, timeout_ms)
        except abi.ZeroError as e:
            if e.code == abi.ZERO_ETIMEDOUT:
                self.t += 1          # the work is queued and will complete
            raise
        self.t += 1
        return self.t

    def bucket_ranges(self, bucket_bytes: int = BUCKET_BYTES_25MIB) -> list:
        count = abi.zero_bucket_count(self.n, self.precision, bucket_bytes)
        return [abi.zero_bucket_range(self.n, self.precision, bucket_bytes, k)
                for k in range(count)]

    # --------------------------------------------------------------- memory --

    def memory_bytes(self, stage: int, rank: int | None = None):
        if rank is None:
            if self.shard_bounds is None:
                return abi.zero_memory_bytes(self.n, self.N, stage, self.precision)
            return max(sum(abi.zero_memory_breakdown_ex(self.n, self.N, stage, self.precision, r,
                                                        self.shard_bounds)) for r in range(self.N))
        return abi.zero_memory_breakdown_ex(self.n, self.N, stage, self.precision, rank,
                                            self.shard_bounds)

    # ------------------------------------------------------- checkpointing --

    def state_dict(self) -> dict:
        d = {"t": self.t}
        for key in ("m", "v", "master"):
            if getattr(self, key) is not None:
                d[key] = getattr(self, key).clone()
        return d

    def load_state_dict(self, d: dict) -> None:
        self.t = int(d["t"])
        for key in ("m", "v", "master"):
            if getattr(self, key) is not None:
                getattr(self, key).copy_(d[key])
