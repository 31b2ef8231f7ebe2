"""GPU parity of the 2:4 training layer (SemiStructuredSparseLinear) against the oracle.

The MLP workload (SparseLinear 512 -> 256, fp16, 4096 tokens, post-ReLU
inputs, W ~ N(0, 0.05), dY ~ N(0, 0.01)) runs forward, backward and the fused
SGD step with re-prune through the layer; Y, dX and dW are compared with the
float64 oracle at the product tolerance, the updated weight, mask and
compressed forms bit for bit.  A GPT-neo FC1-shaped layer (bf16, 16384
tokens) is compared on sampled rows.
"""
import numpy as np
import pytest
import torch

import oracle as o
from structured_sparse_gemm_nm_gb300 import binding as nb
from structured_sparse_gemm_nm_gb300 import inputs
from structured_sparse_gemm_nm_gb300.sparse_linear import SemiStructuredSparseLinear

from gpu_util import DEV, assert_gemm_close, bits_of, ensure_lib, u32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_lib()


def bits(t: torch.Tensor, dtype: str) -> np.ndarray:
    return bits_of(t, dtype, tuple(t.shape))


def check_compressed(layer, W_bits, dtype):
    """The layer's mask and compressed forms equal the oracle's transposable prune of W_bits."""
    out_f, in_f = layer.out_features, layer.in_features
    _, mask, (v, m), (vT, mT) = o.nm_prune_transposable(W_bits, dtype)
    assert np.array_equal(u32(layer.mask, out_f * in_f // 32), o.mask_to_bits(mask).reshape(-1))
    assert np.array_equal(bits_of(layer.vals, dtype, (out_f, in_f // 2)), v)
    assert np.array_equal(bits_of(layer.valsT, dtype, (in_f, out_f // 2)), vT)
    want_tc = o.meta_to_tc_layout(m, out_f, in_f)
    assert np.array_equal(u32(layer.meta, want_tc.size).reshape(want_tc.shape), want_tc)
    want_tcT = o.meta_to_tc_layout(mT, in_f, out_f)
    assert np.array_equal(u32(layer.metaT, want_tcT.size).reshape(want_tcT.shape), want_tcT)
    return mask


def test_mlp_layer_forward_backward_and_fused_step():
    out_f, in_f, T, dt = 256, 512, 4096, "f16"
    W = inputs.normal((out_f, in_f), 0.05, inputs.SEED_W, dt)
    X = inputs.relu_normal((T, in_f), inputs.SEED_X, dt)
    dY = inputs.normal((T, out_f), 0.01, inputs.SEED_DY, dt)
    layer = SemiStructuredSparseLinear(in_f, out_f, torch.float16, DEV, weight=W.to(DEV))
    Xd = X.to(DEV).requires_grad_(True)
    Y = layer(Xd)
    Y.backward(dY.to(DEV))
    torch.cuda.synchronize()

    Wb = inputs.as_numpy_bits(W)
    mask = check_compressed(layer, Wb, dt)
    Wp = o.decode(np.where(mask, Wb, 0).astype(np.uint16), dt)
    Xm, dYm = o.decode(inputs.as_numpy_bits(X), dt), o.decode(inputs.as_numpy_bits(dY), dt)
    assert_gemm_close(Y.detach().cpu().double().numpy(), o.spmm(1.0, Xm, Wp.T), "Y")
    assert_gemm_close(Xd.grad.cpu().double().numpy(), o.spmm(1.0, dYm, Wp), "dX")
    dW_ref = o.masked_weight_grad(dYm, Xm, mask)
    assert_gemm_close(layer.weight.grad.cpu().double().numpy(), dW_ref, "dW")

    # the optimizer's write fused with the re-prune: bit-exact against the oracle's update of the
    # same gradient bits
    lr = 0.5
    G = bits(layer.weight.grad, dt)
    layer.sgd_step_(lr)
    torch.cuda.synchronize()
    W_new = o.sgd_update(Wb, G, lr, dt)
    assert np.array_equal(bits(layer.weight.data, dt), W_new)
    mask2 = check_compressed(layer, W_new, dt)

    # the next step uses the new mask
    layer.weight.grad = None
    Xd.grad = None
    Y2 = layer(Xd)
    torch.cuda.synchronize()
    Wp2 = o.decode(np.where(mask2, W_new, 0).astype(np.uint16), dt)
    assert_gemm_close(Y2.detach().cpu().double().numpy(), o.spmm(1.0, Xm, Wp2.T), "Y after the step")


def test_layer_reprunes_after_an_outside_weight_change():
    out_f, in_f, T = 128, 256, 512
    W = inputs.normal((out_f, in_f), 0.05, 7, "bf16")
    layer = SemiStructuredSparseLinear(in_f, out_f, torch.bfloat16, DEV, weight=W.to(DEV))
    X = inputs.normal((T, in_f), 1.0, 8, "bf16").to(DEV)
    layer(X)
    with torch.no_grad():
        layer.weight.mul_(-2.0)  # an in-place torch update bumps the weight's version
    Y = layer(X)
    torch.cuda.synchronize()
    Wb = bits(layer.weight.data, "bf16")
    mask = check_compressed(layer, Wb, "bf16")
    Wp = o.decode(np.where(mask, Wb, 0).astype(np.uint16), "bf16")
    ref = o.spmm(1.0, o.decode(bits(X, "bf16"), "bf16"), Wp.T)
    assert_gemm_close(Y.detach().cpu().double().numpy(), ref, "Y after an outside update")


def test_gptneo_fc1_layer_sampled_rows():
    out_f, in_f, T, dt = 3072, 768, 16384, "bf16"
    W = inputs.normal((out_f, in_f), 0.02, 11, dt)
    X = inputs.normal((T, in_f), 1.0, 12, dt)
    dY = inputs.normal((T, out_f), 1.0, 13, dt)
    layer = SemiStructuredSparseLinear(in_f, out_f, torch.bfloat16, DEV, weight=W.to(DEV))
    kept = layer.tune_(T, X.to(DEV), dY.to(DEV))  # plan-time search on this token count
    assert set(kept.values()) <= {nb.NM_ALGO_PAIRED, nb.NM_ALGO_SINGLE}
    Xd = X.to(DEV).requires_grad_(True)
    Y = layer(Xd)
    Y.backward(dY.to(DEV))
    torch.cuda.synchronize()
    Wb = inputs.as_numpy_bits(W)
    mask = check_compressed(layer, Wb, dt)
    Wp = o.decode(np.where(mask, Wb, 0).astype(np.uint16), dt)
    rng = np.random.default_rng(3)
    toks = np.sort(rng.choice(T, 128, replace=False))
    Xm, dYm = o.decode(inputs.as_numpy_bits(X), dt), o.decode(inputs.as_numpy_bits(dY), dt)
    assert_gemm_close(Y.detach().cpu().double().numpy()[toks], o.spmm(1.0, Xm[toks], Wp.T), "Y rows")
    assert_gemm_close(Xd.grad.cpu().double().numpy()[toks], o.spmm(1.0, dYm[toks], Wp), "dX rows")
    outs = np.sort(rng.choice(out_f, 64, replace=False))
    dW_ref = o.masked_weight_grad(dYm[:, outs], Xm, mask[outs])
    assert_gemm_close(layer.weight.grad.cpu().double().numpy()[outs], dW_ref, "dW rows")
