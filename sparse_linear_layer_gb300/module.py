"""torch.nn front end: a drop-in replacement for nn.Linear whose weight is
stored only as its non-zeros, with autograd, plus the SET and RigL
schedules that restructure it during training.

  "Beyond Masked Sparsity: SNACK Enables Truly Sparse Neural Networks on
    GPU", abstract and Fig. 1: a drop-in nn.Linear replacement whose weight
    lives as a COO triple, trained with forward / backward passes computed on
    the non-zeros and connections dropped and grown in place.
  "Padded-CSR: A sparse storage format for dynamic sparse training on CPU",
    sec. 8.2: the SparseLinear(in, out, sparsity) layer and the SET(...)
    algorithm object with a step() called once per training step.

Everything numeric runs in libsnk's kernels (through binding.py); this file
only wires them into torch.autograd and keeps the schedule.  The weight's
values are an nn.Parameter (float32, shape [nnz], canonical order), so any
torch optimizer updates them in place; rows and cols are buffers.  The
library borrows all three for the life of the layer.
"""
from __future__ import annotations

import torch

from . import binding, synth


class _SparseLinearFn(torch.autograd.Function):
    @staticmethod
    def forward(ctx, x, values, bias, layer):
        x2 = x.reshape(-1, layer.in_features).contiguous()
        y = torch.empty((x2.shape[0], layer.out_features), dtype=torch.float32, device=x.device)
        binding.snk_forward(layer._h.handle, x2, bias, y)
        ctx.layer = layer
        ctx.has_bias = bias is not None
        ctx.shape = x.shape
        ctx.save_for_backward(x2)
        return y.reshape(*x.shape[:-1], layer.out_features)

    @staticmethod
    def backward(ctx, gy):
        (x2,) = ctx.saved_tensors
        layer = ctx.layer
        gy2 = gy.reshape(-1, layer.out_features).contiguous().float()
        gx = gvalues = gbias = None
        if ctx.needs_input_grad[0]:
            gx = torch.empty_like(x2)
            binding.snk_backward_input(layer._h.handle, gy2, gx)
            gx = gx.reshape(ctx.shape)
        if ctx.needs_input_grad[1] or (ctx.has_bias and ctx.needs_input_grad[2]):
            gvalues = torch.empty_like(layer.values)
            gb = torch.empty(layer.out_features, dtype=torch.float32, device=gy.device) \
                if ctx.has_bias else None
            binding.snk_backward_weight(layer._h.handle, x2, gy2, gvalues, gb)
            gbias = gb if ctx.has_bias and ctx.needs_input_grad[2] else None
            if not ctx.needs_input_grad[1]:
                gvalues = None
        return gx, gvalues, gbias, None


class SparseLinear(torch.nn.Module):
    """y = x W^T + b with W (out x in) kept as its non-zeros only.

    SparseLinear(in_features, out_features, sparsity) draws a uniform random
    support of round(out*in*(1 - sparsity)) positions and values
    N(0, 1/(in*density)); from_triple() binds an existing triple."""

    def __init__(self, in_features: int, out_features: int, sparsity: float, bias: bool = True,
                 seed: int = 0, device=None):
        super().__init__()
        device = torch.device(device if device is not None else "cuda")
        density = 1.0 - sparsity
        nnz = synth.nnz_for(out_features, in_features, 100.0 * sparsity)
        rows, cols = synth.uniform_support(out_features, in_features, nnz, seed)
        std = (1.0 / max(1e-12, in_features * density)) ** 0.5
        values = synth.normal(nnz, std, seed + 1)
        self._bind(in_features, out_features, torch.from_numpy(values).to(device),
                   torch.from_numpy(rows).to(device), torch.from_numpy(cols).to(device), bias)

    @classmethod
    def from_triple(cls, in_features: int, out_features: int, values, rows, cols,
                    bias: bool = True):
        self = cls.__new__(cls)
        torch.nn.Module.__init__(self)
        self._bind(in_features, out_features, values.float().contiguous(),
                   rows.int().contiguous(), cols.int().contiguous(), bias)
        return self

    def _bind(self, in_features, out_features, values, rows, cols, bias):
        self.in_features, self.out_features = in_features, out_features
        self.values = torch.nn.Parameter(values)
        self.register_buffer("rows", rows)
        self.register_buffer("cols", cols)
        self.bias = torch.nn.Parameter(torch.zeros(out_features, device=values.device)) \
            if bias else None
        # sorts the triple in place into canonical order and builds the views
        self._h = binding.SparseLinear(out_features, in_features, self.values.data, self.rows,
                                       self.cols)

    @property
    def nnz(self) -> int:
        return self.values.numel()

    @property
    def topology_version(self) -> int:
        return self._h.topology_version

    def forward(self, x):
        return _SparseLinearFn.apply(x.float(), self.values, self.bias, self)

    @torch.no_grad()
    def prune_regrow(self, zeta: float, seed: int):
        """SET step: drop the fraction zeta of smallest |w|, grow as many at
        seeded uniform positions with value 0 (the values and the support
        are rewritten in place, nnz unchanged)."""
        self._h.prune_regrow(zeta, seed)

    @torch.no_grad()
    def prune_regrow_gradient(self, zeta: float, x, grad_y):
        """RigL step: the same drop, then growth where |grad_y^T x| is largest."""
        x2 = x.reshape(-1, self.in_features).contiguous().float()
        gy2 = grad_y.reshape(-1, self.out_features).contiguous().float()
        self._h.prune_regrow_gradient(zeta, x2, gy2)

    def dense_weight(self):
        """The weight as a dense tensor (for inspection only)."""
        w = torch.zeros(self.out_features, self.in_features, device=self.values.device)
        w[self.rows.long(), self.cols.long()] = self.values.detach()
        return w

    def extra_repr(self) -> str:
        return (f"in_features={self.in_features}, out_features={self.out_features}, "
                f"nnz={self.nnz}, bias={self.bias is not None}")

    def close(self):
        self._h.close()


class SET:
    """Sparse Evolutionary Training schedule: every `every` calls of step(),
    each SparseLinear restructures with drop fraction zeta and seed
    seed0 + (restructure index) (+ 1000003 * layer index).  Optimizer state
    kept per value (momenta) follows slots, not positions: after a
    restructure it belongs to whatever entry now sits in the slot, as with any
    in-place sparse update; reset it if that matters."""

    def __init__(self, layers, zeta: float = 0.3, every: int = 100, seed0: int = 0x5E7):
        self.layers, self.zeta, self.every, self.seed0 = list(layers), zeta, every, seed0
        self.t = 0
        self.restructures = 0

    def step(self):
        self.t += 1
        if self.t % self.every == 0:
            self.restructures += 1
            for i, layer in enumerate(self.layers):
                layer.prune_regrow(self.zeta, self.seed0 + self.restructures + 1000003 * i)
            return True
        return False
