"""GPU parity of activation 2:4 sparsity (SparseActivationLinear) against the oracle.

The activations entering the layer are pruned 2:4 along their features at run
time (one pass: pruned copy, mask, compressed form), the forward product takes
them as the sparse operand, and the backward products are the masked dX and
the dense dW on the pruned activations.  The MLP workload's post-ReLU inputs
(4096 x 512, fp16) are compared in full, a GPT-neo FC2-shaped layer (bf16,
16384 tokens) on sampled rows.
"""
import numpy as np
import pytest
import torch

import oracle as o
from structured_sparse_gemm_nm_gb300 import binding as nb
from structured_sparse_gemm_nm_gb300 import inputs
from structured_sparse_gemm_nm_gb300.sparse_activation import SparseActivationLinear

from gpu_util import DEV, assert_gemm_close, bits_of, dev_bytes, ensure_lib, u32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_lib()


def test_prune_compress_one_pass_matches_oracle():
    rows, cols = 1000, 512
    X = inputs.relu_normal((rows, cols), 21, "bf16")
    Xd = X.to(DEV)
    vb, mb = nb.nm_compressed_size(rows, cols, "bf16", 2, 4, nb.NM_META_TC)
    vals, meta = dev_bytes(vb), dev_bytes(mb)
    Xp = torch.empty_like(Xd)
    mask = torch.empty(rows * cols // 32, dtype=torch.int32, device=DEV)
    nb.nm_prune_compress(Xd, rows, cols, cols, "bf16", 2, 4, Xp, cols, mask, nb.NM_META_TC, vals, meta)
    torch.cuda.synchronize()
    Xb = inputs.as_numpy_bits(X)
    pruned, m = o.nm_prune(Xb, "bf16", 2, 4)
    v, mc = o.nm_compress(Xb, "bf16", 2, 4)
    assert np.array_equal(bits_of(Xp, "bf16", (rows, cols)), pruned)
    assert np.array_equal(u32(mask, rows * cols // 32), o.mask_to_bits(m).reshape(-1))
    assert np.array_equal(bits_of(vals, "bf16", (rows, cols // 2)), v)
    want = o.meta_to_tc_layout(mc, rows, cols)
    assert np.array_equal(u32(meta, want.size).reshape(want.shape), want)


@pytest.mark.parametrize("shape,dtype,sampled", [((4096, 512, 256), "f16", False), ((16384, 3072, 768), "bf16", True)])
def test_activation_sparse_layer_matches_oracle(shape, dtype, sampled):
    T, in_f, out_f = shape
    tdt = torch.float16 if dtype == "f16" else torch.bfloat16
    W = inputs.normal((out_f, in_f), 0.05 if in_f == 512 else 0.02, 31, dtype)
    X = inputs.relu_normal((T, in_f), 32, dtype)
    dY = inputs.normal((T, out_f), 0.01 if in_f == 512 else 1.0, 33, dtype)
    layer = SparseActivationLinear(in_f, out_f, tdt, DEV, weight=W.to(DEV))
    Xd = X.to(DEV).requires_grad_(True)
    Y = layer(Xd)
    Y.backward(dY.to(DEV))
    torch.cuda.synchronize()
    pruned, mask = o.nm_prune(inputs.as_numpy_bits(X), dtype, 2, 4)
    Xp = o.decode(pruned, dtype)
    Wm = o.decode(inputs.as_numpy_bits(W), dtype)
    dYm = o.decode(inputs.as_numpy_bits(dY), dtype)
    rng = np.random.default_rng(9)
    toks = np.sort(rng.choice(T, 256, replace=False)) if sampled else np.arange(T)
    assert_gemm_close(Y.detach().cpu().double().numpy()[toks], o.spmm(1.0, Xp[toks], Wm.T), "Y")
    dX_ref = np.where(mask[toks], o.spmm(1.0, dYm[toks], Wm), 0.0)
    assert_gemm_close(Xd.grad.cpu().double().numpy()[toks], dX_ref, "dX")
    outs = np.sort(rng.choice(out_f, 64, replace=False)) if sampled else np.arange(out_f)
    dW_ref = o.spmm(1.0, dYm[:, outs].T, Xp)
    assert_gemm_close(layer.weight.grad.cpu().double().numpy()[outs], dW_ref, "dW")
