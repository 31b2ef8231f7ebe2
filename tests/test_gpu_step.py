"""One layer of the benchmark's own training step, checked against the oracle.

The step is the one bench.py times: the run-time transposable prune of every
weight on its own stream, the sparse forward products in layer order, the
sparse dX products in reverse order and each masked dW beside them on a third
stream, with the plans searched as in the benchmark.  For the four GPT-neo
linears of one layer (16384 tokens, bf16) Y, dX and dW are compared with the
float64 oracle on sampled rows, and the compressed weights bit for bit.
"""
import numpy as np
import pytest
import torch

import bench
import oracle as o
from structured_sparse_gemm_nm_gb300 import binding as nb
from structured_sparse_gemm_nm_gb300 import inputs

from gpu_util import DEV, assert_gemm_close, bits_of, ensure_lib

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_lib()


def test_one_layer_of_the_bench_step_matches_oracle():
    T = inputs.GPTNEO_TOKENS
    wl = bench.GptNeoTrain(torch, nb, inputs, DEV, layers=1, tokens=T)
    wl.search_plans()
    for L in wl.layers[0]:
        for k in ("Y", "dX", "dW"):
            L[k].fill_(float("nan"))
    torch.cuda.synchronize()
    launches = wl.enqueue_training_step()
    torch.cuda.synchronize()
    # prune, forward and dX: one kernel each; dW: the product, plus the finalize where its K
    # splits are not summed inside it (as the plan reports)
    dw = [nb.nm_spmm_plan_launches(wl.p_dw[j]) for j in range(4)]
    assert launches == 4 + 4 + 4 + sum(dw)
    # a product whose K is not split, or split in two on paired CTAs, is one launch; other splits
    # add the finalize
    assert all(x in (1, 2) for x in dw)
    rng = np.random.default_rng(17)
    for j, (name, out_f, in_f) in enumerate(wl.linears):
        L = wl.layers[0][j]
        Wb = bits_of(L["W"], "bf16", (out_f, in_f))
        _, mask, (v, _), (vT, _) = o.nm_prune_transposable(Wb, "bf16")
        assert np.array_equal(bits_of(L["vals"], "bf16", (out_f, in_f // 2)), v), name
        assert np.array_equal(bits_of(L["valsT"], "bf16", (in_f, out_f // 2)), vT), name
        Wp = o.decode(np.where(mask, Wb, 0).astype(np.uint16), "bf16")
        X = o.decode(bits_of(L["X"], "bf16", (T, in_f)), "bf16")
        dY = o.decode(bits_of(L["dY"], "bf16", (T, out_f)), "bf16")
        toks = np.sort(rng.choice(T, 128, replace=False))
        Y = L["Y"].cpu().double().numpy()
        dX = L["dX"].cpu().double().numpy()
        assert_gemm_close(Y[toks], o.spmm(1.0, X[toks], Wp.T), f"{name} Y")
        assert_gemm_close(dX[toks], o.spmm(1.0, dY[toks], Wp), f"{name} dX")
        outs = np.sort(rng.choice(out_f, 64, replace=False))
        dW = L["dW"].cpu().double().numpy()
        assert_gemm_close(dW[outs], o.masked_weight_grad(dY[:, outs], X, mask[outs]), f"{name} dW")
