"""A linear layer whose input activations are pruned 2:4 at run time.

PyTorch issue #126420's maintainer reply names activation sparsity beside
weight sparsity: the 2:4 pattern is imposed on the activations that enter a
linear layer (typically after a ReLU-like nonlinearity, where many are already
zero), and the sparse tensor cores take the activations as the sparse operand.
Every step runs in the CUDA library through its C ABI:

* ``nm_prune_compress`` reads X once and writes the pruned activations (the
  greedy 2:4 rule along the features: the two largest |x| of every four, ties
  to the lower position), their bit mask and their compressed form;
* forward ``Y = X_sp W^T`` is the 2:4 sparse product with A = compressed X
  (M = tokens, K = in features) and B = W, Y written row-major;
* backward ``dX = mask_X * (dY W)``: the pruned activations pass gradient only
  at their kept positions, a masked dense product;
* backward ``dW = dY^T X_sp``: the dense product on the pruned activations
  (a masked dense product with no mask).

W stays dense.  Inputs must be contiguous 16-bit CUDA tensors, the feature
count a multiple of 32; there is no fallback.
"""
from __future__ import annotations

import torch

from . import binding as nb

_DTYPES = {torch.float16: "f16", torch.bfloat16: "bf16"}


class _ActPlans:
    def __init__(self, out_f: int, in_f: int, tokens: int, dt: str, device):
        # forward: A = compressed X (tokens x in), B = W stored out x in (N x K), D = Y row-major (tokens x out)
        self.fwd = nb.nm_spmm_plan(nb.make_desc(M=tokens, N=out_f, K=in_f, ab_type=dt, cd_type=dt, ldb=in_f,
                                                order_cd=nb.NM_ROW, ldd=out_f))
        # dX: A = dY (tokens x out, K-major), B = W (out x in = K x N row-major), mask of X, D = dX (tokens x in)
        self.dx = nb.nm_spmm_plan(nb.make_desc(M=tokens, N=in_f, K=out_f, mode=nb.NM_SPMM_DENSE_MASKED, ab_type=dt,
                                               cd_type=dt, order_a=nb.NM_ROW, order_b=nb.NM_ROW, order_cd=nb.NM_ROW,
                                               lda=out_f, ldb=in_f, ldd=in_f, meta_layout=nb.NM_META_CANONICAL))
        # dW: A = dY (tokens x out = K x M, M-major), B = X_sp (tokens x in = K x N), no mask, D = dW (out x in)
        self.dw = nb.nm_spmm_plan(nb.make_desc(M=out_f, N=in_f, K=tokens, mode=nb.NM_SPMM_DENSE_MASKED, ab_type=dt,
                                               cd_type=dt, order_a=nb.NM_COL, order_b=nb.NM_ROW, order_cd=nb.NM_ROW,
                                               lda=out_f, ldb=in_f, ldd=in_f, meta_layout=nb.NM_META_CANONICAL))
        self.ws = []
        for p in (self.dx, self.dw):
            b = nb.nm_spmm_plan_workspace(p)
            self.ws.append((torch.empty(max(16, b), dtype=torch.uint8, device=device) if b else None, b))


class SparseActivationFunction(torch.autograd.Function):
    @staticmethod
    def forward(ctx, X: torch.Tensor, weight: torch.Tensor, layer: "SparseActivationLinear"):
        T, in_f = X.shape
        dt = layer._dt
        plans = layer._plans_for(T)
        Xp = torch.empty_like(X)
        mask = torch.empty(T * in_f // 32, dtype=torch.int32, device=X.device)
        vb, mb = nb.nm_compressed_size(T, in_f, dt, 2, 4, nb.NM_META_TC)
        vals = torch.empty(max(16, vb), dtype=torch.uint8, device=X.device)
        meta = torch.empty(max(16, mb), dtype=torch.uint8, device=X.device)
        nb.nm_prune_compress(X, T, in_f, in_f, dt, 2, 4, Xp, in_f, mask, nb.NM_META_TC, vals, meta)
        Y = torch.empty((T, layer.out_features), dtype=X.dtype, device=X.device)
        nb.nm_spmm(plans.fwd, 1.0, vals, meta, weight.detach(), 0.0, None, Y)
        ctx.save_for_backward(Xp, mask, weight)
        ctx.layer = layer
        return Y

    @staticmethod
    def backward(ctx, dY: torch.Tensor):
        Xp, mask, weight = ctx.saved_tensors
        layer = ctx.layer
        if not dY.is_contiguous():
            raise ValueError("SparseActivationLinear needs a contiguous output gradient")
        plans = layer._plans_for(Xp.shape[0])
        dX = dW = None
        if ctx.needs_input_grad[0]:
            dX = torch.empty_like(Xp)
            ws, wsb = plans.ws[0]
            nb.nm_spmm(plans.dx, 1.0, dY, mask, weight.detach(), 0.0, None, dX, ws, wsb)
        if ctx.needs_input_grad[1]:
            dW = torch.empty((layer.out_features, layer.in_features), dtype=Xp.dtype, device=Xp.device)
            ws, wsb = plans.ws[1]
            nb.nm_spmm(plans.dw, 1.0, dY, None, Xp, 0.0, None, dW, ws, wsb)
        return dX, dW, None


class SparseActivationLinear(torch.nn.Module):
    """Bias-free linear layer whose input is pruned 2:4 along its features at run time."""

    def __init__(self, in_features: int, out_features: int, dtype=torch.bfloat16, device="cuda", weight=None):
        super().__init__()
        if dtype not in _DTYPES:
            raise ValueError("SparseActivationLinear takes float16 or bfloat16")
        if in_features % 32 or out_features % 8:
            raise ValueError("in_features must be a multiple of 32 and out_features of 8")
        device = torch.device(device)
        if device.type != "cuda":
            raise ValueError("SparseActivationLinear runs on a CUDA device only")
        self.in_features, self.out_features = in_features, out_features
        self._dt = _DTYPES[dtype]
        if weight is None:
            weight = torch.empty((out_features, in_features), dtype=dtype, device=device)
            torch.nn.init.kaiming_uniform_(weight, a=5 ** 0.5)
        elif tuple(weight.shape) != (out_features, in_features) or weight.dtype != dtype:
            raise ValueError("weight must be out_features x in_features of the layer's dtype")
        self.weight = torch.nn.Parameter(weight.detach().to(device).contiguous())
        self._plans = {}

    def _plans_for(self, tokens: int) -> _ActPlans:
        p = self._plans.get(tokens)
        if p is None:
            p = self._plans[tokens] = _ActPlans(self.out_features, self.in_features, tokens, self._dt,
                                                self.weight.device)
        return p

    def forward(self, x: torch.Tensor) -> torch.Tensor:
        if x.device.type != "cuda" or x.dtype != self.weight.dtype:
            raise ValueError("input must be a CUDA tensor of the layer's dtype")
        if x.shape[-1] != self.in_features or not x.is_contiguous():
            raise ValueError("input must be contiguous with in_features features")
        X2 = x.view(-1, self.in_features)
        Y = SparseActivationFunction.apply(X2, self.weight, self)
        return Y.view(*x.shape[:-1], self.out_features)

    def extra_repr(self) -> str:
        return f"in_features={self.in_features}, out_features={self.out_features}, activations=2:4 at run time"
