"""A bias-free linear layer trained with a transposable 2:4 mask.

This is the training-side use of the library that PyTorch issue #126420's
maintainer reply describes: a drop-in replacement for ``nn.Linear`` built on a
``torch.autograd.Function``, whose weight mask is 2:4 in 4x4 tiles so that the
forward product ``W x`` and the backward product ``W^T dL/dy`` both run on the
sparse tensor cores, with the weight pruned and compressed at run time by fast
kernels.  Every step runs in the CUDA library through its C ABI:

* the run-time prune (``nm_prune_transposable``) derives, from the dense master
  weight, the bit mask and the compressed forms of ``W`` and ``W^T``
  (tensor-core metadata);
* forward ``Y = X W^T`` is the 2:4 sparse product with A = compressed ``W``;
* backward ``dX = dY W`` is the 2:4 sparse product with A = compressed
  ``W^T``, and ``dW = mask * (dY^T X)`` is the masked dense product;
* ``sgd_step_`` is the optimizer's weight write fused with the re-prune
  (``nm_sgd_prune_transposable``): ``W <- W - lr * dW`` and the new mask and
  compressed forms, in one pass over the weight.

PyTorch provides the tensors, the current stream and the autograd graph; it
computes nothing here.  Inputs must be contiguous 16-bit CUDA tensors; there is
no fallback.
"""
from __future__ import annotations

import torch

from . import binding as nb

_DTYPES = {torch.float16: "f16", torch.bfloat16: "bf16"}


class _Plans:
    """The three product plans of one token count, and the weight-gradient workspace."""

    def __init__(self, out_f: int, in_f: int, tokens: int, dt: str, device):
        self.fwd = nb.nm_spmm_plan(nb.make_desc(M=out_f, N=tokens, K=in_f, ab_type=dt, cd_type=dt, ldb=in_f,
                                                ldd=out_f))
        self.dx = nb.nm_spmm_plan(nb.make_desc(M=in_f, N=tokens, K=out_f, ab_type=dt, cd_type=dt, ldb=out_f,
                                               ldd=in_f))
        self.dw = nb.nm_spmm_plan(nb.make_desc(M=out_f, N=in_f, K=tokens, mode=nb.NM_SPMM_DENSE_MASKED, ab_type=dt,
                                               cd_type=dt, order_a=nb.NM_COL, order_b=nb.NM_ROW, order_cd=nb.NM_ROW,
                                               lda=out_f, ldb=in_f, ldd=in_f, meta_layout=nb.NM_META_CANONICAL))
        self.ws_bytes = nb.nm_spmm_plan_workspace(self.dw)
        self.ws = torch.empty(max(16, self.ws_bytes), dtype=torch.uint8, device=device) if self.ws_bytes else None


class SparseLinearFunction(torch.autograd.Function):
    """Y = X W^T with the layer's compressed weight; dX and the masked dW in backward."""

    @staticmethod
    def forward(ctx, X: torch.Tensor, weight: torch.Tensor, layer: "SemiStructuredSparseLinear"):
        plans = layer._plans_for(X.shape[0])
        Y = torch.empty((X.shape[0], layer.out_features), dtype=X.dtype, device=X.device)
        nb.nm_spmm(plans.fwd, 1.0, layer.vals, layer.meta, X, 0.0, None, Y)
        ctx.save_for_backward(X)
        ctx.layer = layer
        return Y

    @staticmethod
    def backward(ctx, dY: torch.Tensor):
        (X,) = ctx.saved_tensors
        layer = ctx.layer
        if not dY.is_contiguous():
            raise ValueError("SemiStructuredSparseLinear needs a contiguous output gradient")
        plans = layer._plans_for(X.shape[0])
        dX = dW = None
        if ctx.needs_input_grad[0]:
            dX = torch.empty_like(X)
            nb.nm_spmm(plans.dx, 1.0, layer.valsT, layer.metaT, dY, 0.0, None, dX)
        if ctx.needs_input_grad[1]:
            dW = torch.empty((layer.out_features, layer.in_features), dtype=X.dtype, device=X.device)
            nb.nm_spmm(plans.dw, 1.0, dY, layer.mask, X, 0.0, None, dW, plans.ws, plans.ws_bytes)
        return dX, dW, None


class SemiStructuredSparseLinear(torch.nn.Module):
    """``nn.Linear`` without bias whose weight trains under a transposable 2:4 mask.

    The dense master weight is a ``Parameter``; the mask and the compressed
    forms of ``W`` and ``W^T`` are buffers derived from it at run time (again
    whenever the weight changed since the last prune).  Use ``sgd_step_`` for
    the fused update, or any optimizer followed by the next forward's re-prune.
    Gradients are produced, not accumulated: clear them with ``set_to_none``.
    ``in_features`` and ``out_features`` must be multiples of 32 (the
    tensor-core metadata layout of ``W`` and of ``W^T``).
    """

    def __init__(self, in_features: int, out_features: int, dtype=torch.bfloat16, device="cuda", weight=None):
        super().__init__()
        if dtype not in _DTYPES:
            raise ValueError("SemiStructuredSparseLinear takes float16 or bfloat16 weights")
        if in_features % 32 or out_features % 32:
            raise ValueError("in_features and out_features must be multiples of 32")
        self.in_features, self.out_features = in_features, out_features
        self._dt = _DTYPES[dtype]
        device = torch.device(device)
        if device.type != "cuda":
            raise ValueError("SemiStructuredSparseLinear runs on a CUDA device only")
        if weight is None:
            weight = torch.empty((out_features, in_features), dtype=dtype, device=device)
            torch.nn.init.kaiming_uniform_(weight, a=5 ** 0.5)
        elif tuple(weight.shape) != (out_features, in_features) or weight.dtype != dtype:
            raise ValueError("weight must be out_features x in_features of the layer's dtype")
        self.weight = torch.nn.Parameter(weight.detach().to(device).contiguous())
        vb, mb = nb.nm_compressed_size(out_features, in_features, self._dt, 2, 4, nb.NM_META_TC)
        vbT, mbT = nb.nm_compressed_size(in_features, out_features, self._dt, 2, 4, nb.NM_META_TC)

        def buf(nbytes):
            return torch.empty(max(16, nbytes), dtype=torch.uint8, device=device)

        self.register_buffer("vals", buf(vb), persistent=False)
        self.register_buffer("meta", buf(mb), persistent=False)
        self.register_buffer("valsT", buf(vbT), persistent=False)
        self.register_buffer("metaT", buf(mbT), persistent=False)
        self.register_buffer("mask", torch.empty(out_features * in_features // 32, dtype=torch.int32, device=device),
                             persistent=False)
        self._plans = {}
        self._pruned_version = None

    @classmethod
    def from_linear(cls, linear: torch.nn.Linear) -> "SemiStructuredSparseLinear":
        if linear.bias is not None:
            raise ValueError("the sparse layer has no bias")
        return cls(linear.in_features, linear.out_features, linear.weight.dtype, linear.weight.device,
                   weight=linear.weight.data)

    def _plans_for(self, tokens: int) -> _Plans:
        p = self._plans.get(tokens)
        if p is None:
            p = self._plans[tokens] = _Plans(self.out_features, self.in_features, tokens, self._dt,
                                             self.weight.device)
        return p

    def prune_(self) -> None:
        """Run-time transposable prune and compression of the current weight."""
        W = self.weight.data
        nb.nm_prune_transposable(W, self.out_features, self.in_features, self.in_features, self._dt, None, 0,
                                 self.mask, self.vals, self.meta, self.valsT, self.metaT, nb.NM_META_TC)
        self._pruned_version = self.weight._version

    def sgd_step_(self, lr: float) -> None:
        """W <- W - lr * W.grad and the re-prune of the updated weight, in one library pass."""
        g = self.weight.grad
        if g is None:
            raise RuntimeError("no gradient: run backward first")
        if not g.is_contiguous():
            raise ValueError("the weight gradient must be contiguous")
        W = self.weight.data
        nb.nm_sgd_prune_transposable(W, g, lr, self.out_features, self.in_features, self.in_features,
                                     self.in_features, self._dt, self.mask, self.vals, self.meta, self.valsT,
                                     self.metaT, nb.NM_META_TC)
        self._pruned_version = self.weight._version

    def tune_(self, tokens: int, X: torch.Tensor, dY: torch.Tensor) -> dict:
        """Plan-time algorithm search of this token count's three products on sample operands
        (synchronises the stream; call outside graph capture).  Returns the kernels kept."""
        if self._pruned_version != self.weight._version:
            self.prune_()
        p = self._plans_for(tokens)
        Y = torch.empty((tokens, self.out_features), dtype=X.dtype, device=X.device)
        dX = torch.empty((tokens, self.in_features), dtype=X.dtype, device=X.device)
        dW = torch.empty((self.out_features, self.in_features), dtype=X.dtype, device=X.device)
        return {"fwd": nb.nm_spmm_search(p.fwd, 1.0, self.vals, self.meta, X, 0.0, None, Y),
                "dx": nb.nm_spmm_search(p.dx, 1.0, self.valsT, self.metaT, dY, 0.0, None, dX),
                "dw": nb.nm_spmm_search(p.dw, 1.0, dY, self.mask, X, 0.0, None, dW, p.ws, p.ws_bytes)}

    def forward(self, x: torch.Tensor) -> torch.Tensor:
        if x.device.type != "cuda" or x.dtype != self.weight.dtype:
            raise ValueError("input must be a CUDA tensor of the layer's dtype")
        if x.shape[-1] != self.in_features:
            raise ValueError(f"input has {x.shape[-1]} features, the layer {self.in_features}")
        if not x.is_contiguous():
            raise ValueError("SemiStructuredSparseLinear needs a contiguous input")
        if self._pruned_version != self.weight._version:
            self.prune_()
        X2 = x.view(-1, self.in_features)
        Y = SparseLinearFunction.apply(X2, self.weight, self)
        return Y.view(*x.shape[:-1], self.out_features)

    def extra_repr(self) -> str:
        return f"in_features={self.in_features}, out_features={self.out_features}, sparsity=2:4 transposable"
