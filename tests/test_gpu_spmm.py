"""GPU parity of the products against the CPU oracle (float64 reference).

Sparse 2:4 on tensor cores (forward and the transposed backward operand),
the masked dense weight gradient, and the CUDA-core N:M gather.  Small shapes
span several tiles with ragged tails and are compared in full; the workloads'
full sizes run in the launch configuration the benchmark uses and are
compared on sampled rows that the oracle computes one by one.
"""
import numpy as np
import pytest
import torch

import oracle as o
from structured_sparse_gemm_nm_gb300 import binding as nb
from structured_sparse_gemm_nm_gb300 import inputs

from gpu_util import DEV, assert_gemm_close, bits_of, dev_bytes, ensure_lib, to_dev_bits

TORCH_OUT = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_lib()


def compress_on_gpu(Wd, M, K, dtype, layout=nb.NM_META_TC, transpose=0):
    rl, cl = (K, M) if transpose else (M, K)
    vb, mb = nb.nm_compressed_size(rl, cl, dtype, 2, 4, layout)
    vals, meta = dev_bytes(vb), dev_bytes(mb)
    ld = Wd.shape[1] if Wd.dim() == 2 else K
    nb.nm_compress(Wd, M, K, ld, dtype, 2, 4, transpose, layout, vals, meta)
    return vals, meta


def sample_rows(M, count, seed):
    if M <= count:
        return np.arange(M)
    return np.sort(np.random.default_rng(seed).choice(M, size=count, replace=False))


SPARSE_CASES = [
    # M, N, K, dtype, order_cd, alpha, beta, sampled
    (64, 32, 128, "f16", nb.NM_COL, 1.0, 0.0, False),      # tiny round trip
    (256, 4096, 512, "f16", nb.NM_COL, 1.0, 0.0, False),   # SparseLinear forward
    (512, 4096, 256, "f16", nb.NM_COL, 1.0, 0.0, False),   # its backward (W^T operand shape)
    (200, 300, 224, "bf16", nb.NM_COL, 1.0, 0.0, False),   # ragged M, N and K % 128
    (136, 72, 96, "f16", nb.NM_ROW, 2.0, 0.5, False),      # row-major D, alpha/beta
    (384, 264, 640, "bf16", nb.NM_ROW, -0.5, 1.0, False),
    (128, 128, 32, "f16", nb.NM_COL, 1.0, 0.25, False),    # a single MMA k-step
    (264, 200, 160, "f16", nb.NM_ROW, 1.5, 0.0, False),    # row-major D through the bulk-store path
    (96, 40, 32, "bf16", nb.NM_COL, 1.0, 0.0, False),      # one partial tile, one k-step
    # paired CTAs, row-major 16-bit D without C: 32 x 32 blocks staged for TMA stores
    (256, 200, 224, "bf16", nb.NM_ROW, 0.5, 0.0, False),   # ragged N, alpha applied
    (200, 328, 96, "f16", nb.NM_ROW, 1.0, 0.0, False),     # ragged M inside the pair
    (512, 4096, 512, "bf16", nb.NM_ROW, 1.0, 0.0, False),  # several tiles per cluster
    (1024, 4096, 1024, "f16", nb.NM_COL, 1.0, 0.0, True),  # BERT-Large shapes
    (4096, 4096, 1024, "f16", nb.NM_COL, 1.0, 0.0, True),
    (1024, 4096, 4096, "f16", nb.NM_COL, 1.0, 0.0, True),
    (3072, 16384, 768, "bf16", nb.NM_COL, 1.0, 0.0, True),  # GPT-neo FC1 forward
    (768, 16384, 3072, "bf16", nb.NM_COL, 1.0, 0.0, True),  # GPT-neo FC1 backward (dX)
    (2304, 16384, 768, "bf16", nb.NM_COL, 1.0, 0.0, True),  # GPT-neo QKV forward
    (768, 16384, 2304, "bf16", nb.NM_COL, 1.0, 0.0, True),  # GPT-neo QKV backward (dX)
    (768, 16384, 768, "bf16", nb.NM_COL, 1.0, 0.0, True),   # GPT-neo O forward and dX
]

# Every case runs with the library's default (paired CTAs when M spans an even number of
# 128-row blocks, else single CTAs); the even-block cases also run on single CTAs.
SINGLE_CASES = [c for c in SPARSE_CASES if ((c[0] + 127) // 128) % 2 == 0 and not c[7]] + \
    [(3072, 16384, 768, "bf16", nb.NM_COL, 1.0, 0.0, True)]
# an fp32 D (and C) from 16-bit inputs
F32_CASES = [
    (256, 4096, 512, "bf16", nb.NM_COL, 1.0, 0.0, False, "f32"),
    (200, 300, 224, "f16", nb.NM_ROW, 0.5, -1.5, False, "f32"),
    (384, 264, 640, "bf16", nb.NM_COL, 2.0, 1.0, False, "f32"),
    # beta = 0 on paired CTAs: the fp32 epilogue that hands each half back before storing,
    # row-major (16-byte row stores, ragged N) and column-major with a ragged tail
    (256, 200, 224, "bf16", nb.NM_ROW, 0.5, 0.0, False, "f32"),
    (512, 328, 96, "f16", nb.NM_COL, -1.0, 0.0, False, "f32"),
]


@pytest.mark.parametrize("M,N,K,dtype,order_cd,alpha,beta,sampled,algo,cd",
                         [c + (nb.NM_ALGO_DEFAULT, None) for c in SPARSE_CASES] +
                         [c + (nb.NM_ALGO_SINGLE, None) for c in SINGLE_CASES] +
                         [c[:8] + (a, c[8]) for c in F32_CASES for a in (nb.NM_ALGO_DEFAULT, nb.NM_ALGO_SINGLE)])
def test_sparse_tc_matches_oracle(M, N, K, dtype, order_cd, alpha, beta, sampled, algo, cd):
    cd = cd or dtype
    std = 0.02 if K >= 512 else 0.5
    W = inputs.normal((M, K), std, inputs.SEED_W + M, dtype)
    X = inputs.normal((N, K), 1.0, inputs.SEED_X + N, dtype)  # B stored N x K
    Wd, Xd = W.to(DEV), X.to(DEV)
    vals, meta = compress_on_gpu(Wd, M, K, dtype)
    cd_shape = (M, N) if order_cd == nb.NM_ROW else (N, M)
    ld = cd_shape[1]
    C = inputs.normal(cd_shape, 1.0, inputs.SEED_C, "f32" if cd == "f32" else dtype).to(DEV) if beta != 0 else None
    D = torch.full(cd_shape, float("nan"), dtype=TORCH_OUT[cd], device=DEV)
    plan = nb.nm_spmm_plan(nb.make_desc(M=M, N=N, K=K, ab_type=dtype, cd_type=cd, ldb=K,
                                        ldc=ld if C is not None else 0, ldd=ld, order_cd=order_cd, algo=algo))
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    nb.nm_spmm(plan, alpha, vals, meta, Xd, beta, C, D, d_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    Wb = inputs.as_numpy_bits(W)
    A = o.decode(o.nm_prune(Wb, dtype, 2, 4)[0], dtype)
    Bm = o.decode(inputs.as_numpy_bits(X), dtype).T  # K x N
    got = D.cpu().double().numpy()
    got = got if order_cd == nb.NM_ROW else got.T  # M x N
    Cm = None
    if C is not None:
        Cm = C.cpu().double().numpy()
        Cm = Cm if order_cd == nb.NM_ROW else Cm.T
    rows = sample_rows(M, 256, seed=M + N) if sampled else np.arange(M)
    ref = o.spmm(alpha, A[rows], Bm, beta, Cm[rows] if Cm is not None else None)
    assert_gemm_close(got[rows], ref, f"sparse {M}x{N}x{K} {dtype}")


def test_sparse_backward_uses_transposable_compressed_wt():
    """dX^T = W^T dY^T with the W^T operand from the transposable prune (MLP layer 512 -> 256)."""
    out_f, in_f, T = 256, 512, 4096
    W = inputs.normal((out_f, in_f), 0.05, inputs.SEED_W, "f16")
    dY = inputs.normal((T, out_f), 0.01, inputs.SEED_DY, "f16")
    Wd, dYd = W.to(DEV), dY.to(DEV)
    vb, mb = nb.nm_compressed_size(in_f, out_f, "f16", 2, 4, nb.NM_META_TC)
    valsT, metaT = dev_bytes(vb), dev_bytes(mb)
    nb.nm_prune_transposable(Wd, out_f, in_f, in_f, "f16", valsT=valsT, metaT=metaT, layout=nb.NM_META_TC)
    dX = torch.empty((T, in_f), dtype=torch.float16, device=DEV)
    plan = nb.nm_spmm_plan(nb.make_desc(M=in_f, N=T, K=out_f, ab_type="f16", cd_type="f16", ldb=out_f, ldd=in_f))
    nb.nm_spmm(plan, 1.0, valsT, metaT, dYd, 0.0, None, dX)
    torch.cuda.synchronize()
    pruned = o.nm_prune_transposable(inputs.as_numpy_bits(W), "f16")[0]
    ref = o.spmm(1.0, o.decode(pruned, "f16").T, o.decode(inputs.as_numpy_bits(dY), "f16").T)  # in x T
    assert_gemm_close(dX.cpu().double().numpy().T, ref, "dX")


DENSE_CASES = [
    # M (out), N (in), K (tokens), dtype, sampled, alpha, beta
    (256, 512, 4096, "f16", False, 1.0, 0.0),    # SparseLinear 512 -> 256 weight gradient
    (104, 200, 96, "bf16", False, 1.0, 0.0),     # ragged
    (136, 72, 1000, "f16", False, 1.0, 0.0),     # K not a multiple of the stage
    (136, 72, 1000, "f16", False, 0.5, -1.0),    # gradient accumulation into C
    (264, 136, 1000, "bf16", False, 0.5, -1.0),  # ragged, even row blocks, accumulation into C
    (512, 520, 192, "f16", False, 1.0, 0.0),     # no K split, ragged N
    (3072, 768, 16384, "bf16", True, 1.0, 0.0),  # GPT-neo FC1 dW
    (768, 3072, 16384, "bf16", True, 1.0, 0.0),  # GPT-neo FC2 dW
    (2304, 768, 16384, "bf16", True, 1.0, 0.0),  # GPT-neo QKV dW
    (768, 768, 16384, "bf16", True, 1.0, 0.0),   # GPT-neo O dW
]
DENSE_SINGLE = [c for c in DENSE_CASES if not c[4]]


@pytest.mark.parametrize("M,N,K,dtype,sampled,alpha,beta,algo,cd",
                         [c + (nb.NM_ALGO_DEFAULT, None) for c in DENSE_CASES] +
                         [c + (nb.NM_ALGO_SINGLE, None) for c in DENSE_SINGLE] +
                         [(256, 512, 4096, "bf16", False, 1.0, 0.0, a, "f32") for a in (0, 2)] +
                         [(264, 136, 1000, "f16", False, 0.5, -1.0, a, "f32") for a in (0, 2)] +
                         # two K splits on paired CTAs: summed in the product, fp32 D with C
                         [(136, 72, 1000, "bf16", False, 0.5, -1.0, 0, "f32")] +
                         [(512, 520, 192, "bf16", False, 2.0, 0.0, a, "f32") for a in (0, 2)])
def test_masked_weight_grad_matches_oracle(M, N, K, dtype, sampled, alpha, beta, algo, cd):
    cd = cd or dtype
    dY = inputs.normal((K, M), 1.0, inputs.SEED_DY + K, dtype)   # tokens x out
    X = inputs.normal((K, N), 1.0, inputs.SEED_X + K, dtype)     # tokens x in
    W = inputs.normal((M, N), 0.02, inputs.SEED_W, dtype)
    pruned, mask_ref = o.nm_prune(inputs.as_numpy_bits(W), dtype, 2, 4)
    bits = torch.from_numpy(o.mask_to_bits(mask_ref).view(np.int32)).to(DEV)
    dW = torch.full((M, N), float("nan"), dtype=TORCH_OUT[cd], device=DEV)
    C = inputs.normal((M, N), 1.0, inputs.SEED_C, cd) if beta != 0 else None
    plan = nb.nm_spmm_plan(nb.make_desc(M=M, N=N, K=K, mode=nb.NM_SPMM_DENSE_MASKED, ab_type=dtype, cd_type=cd,
                                        order_a=nb.NM_COL, order_b=nb.NM_ROW, order_cd=nb.NM_ROW, lda=M, ldb=N,
                                        ldc=N if C is not None else 0, ldd=N, meta_layout=nb.NM_META_CANONICAL,
                                        algo=algo))
    ws_bytes = nb.nm_spmm_plan_workspace(plan)
    ws = dev_bytes(ws_bytes) if ws_bytes else None
    nb.nm_spmm(plan, alpha, dY.to(DEV), bits, X.to(DEV), beta, C.to(DEV) if C is not None else None, dW, ws, ws_bytes)
    torch.cuda.synchronize()
    rows = sample_rows(M, 128, seed=K) if sampled else np.arange(M)
    dYm = o.decode(inputs.as_numpy_bits(dY), dtype)
    Xm = o.decode(inputs.as_numpy_bits(X), dtype)
    ref = alpha * o.masked_weight_grad(dYm[:, rows], Xm, mask_ref[rows])
    if C is not None:
        ref = ref + beta * C.double().numpy()[rows]
    assert_gemm_close(dW.cpu().double().numpy()[rows], ref, f"dW {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K,beta", [(136, 72, 1000, 0.0), (136, 72, 1000, 2.0), (768, 768, 16384, 0.0)])
def test_masked_weight_grad_column_major(M, N, K, beta):
    """Column-major dW: two K splits summed in the paired product (with and without C), and the
    O dW shape's eight splits summed by the separate finalize."""
    dtype = "bf16"
    dY = inputs.normal((K, M), 1.0, inputs.SEED_DY + K, dtype)
    X = inputs.normal((K, N), 1.0, inputs.SEED_X + K, dtype)
    W = inputs.normal((M, N), 0.02, inputs.SEED_W, dtype)
    _, mask_ref = o.nm_prune(inputs.as_numpy_bits(W), dtype, 2, 4)
    bits = torch.from_numpy(o.mask_to_bits(mask_ref).view(np.int32)).to(DEV)
    dWt = torch.full((N, M), float("nan"), dtype=torch.bfloat16, device=DEV)  # dW column-major: [N][M]
    C = inputs.normal((N, M), 1.0, inputs.SEED_C, dtype) if beta != 0 else None
    plan = nb.nm_spmm_plan(nb.make_desc(M=M, N=N, K=K, mode=nb.NM_SPMM_DENSE_MASKED, ab_type=dtype, cd_type=dtype,
                                        order_a=nb.NM_COL, order_b=nb.NM_ROW, order_cd=nb.NM_COL, lda=M, ldb=N,
                                        ldc=M if C is not None else 0, ldd=M, meta_layout=nb.NM_META_CANONICAL))
    ws_bytes = nb.nm_spmm_plan_workspace(plan)
    ws = dev_bytes(ws_bytes) if ws_bytes else None
    nb.nm_spmm(plan, 1.0, dY.to(DEV), bits, X.to(DEV), beta, C.to(DEV) if C is not None else None, dWt, ws, ws_bytes)
    torch.cuda.synchronize()
    rows = sample_rows(M, 128, seed=K) if M > 512 else np.arange(M)
    dYm = o.decode(inputs.as_numpy_bits(dY), dtype)
    Xm = o.decode(inputs.as_numpy_bits(X), dtype)
    ref = o.masked_weight_grad(dYm[:, rows], Xm, mask_ref[rows])
    if C is not None:
        ref = ref + beta * C.double().numpy().T[rows]
    assert_gemm_close(dWt.cpu().double().numpy().T[rows], ref, f"dW col-major {M}x{N}x{K}")


@pytest.mark.parametrize("n", [4, 8, 16])
@pytest.mark.parametrize("batch", [1, 8])
def test_nm_gather_gemv_matches_oracle(n, batch):
    M = K = 4096
    W = inputs.normal((M, K), 0.02, inputs.SEED_W, "f16")
    x = inputs.normal((batch, K), 1.0, inputs.SEED_VEC, "f16")
    Wd = W.to(DEV)
    vb, mb = nb.nm_compressed_size(M, K, "f16", n, 32)
    vals, idx = dev_bytes(vb), dev_bytes(mb)
    nb.nm_compress(Wd, M, K, K, "f16", n, 32, 0, nb.NM_META_CANONICAL, vals, idx)
    y = torch.empty((batch, M), dtype=torch.float16, device=DEV)
    plan = nb.nm_spmm_plan(nb.make_desc(M=M, N=batch, K=K, n=n, m=32, ab_type="f16", cd_type="f16", ldb=K, ldd=M,
                                        meta_layout=nb.NM_META_CANONICAL))
    nb.nm_spmm(plan, 1.0, vals, idx, x.to(DEV), 0.0, None, y)
    torch.cuda.synchronize()
    A = o.decode(o.nm_prune(inputs.as_numpy_bits(W), "f16", n, 32)[0], "f16")
    ref = o.spmm(1.0, A, o.decode(inputs.as_numpy_bits(x), "f16").T)
    assert_gemm_close(y.cpu().double().numpy().T, ref, f"gemv n={n} b={batch}")


@pytest.mark.parametrize("batch", [1, 8])
def test_gather_many_rows_per_warp(batch):
    # more rows than warps in the whole-wave grid: every warp takes several interleaved rows
    M, K, n, m = 40000 + 3, 64, 8, 32
    W = inputs.normal((M, K), 0.1, 12, "f16")
    x = inputs.normal((batch, K), 1.0, 13, "f16")
    vb, mb = nb.nm_compressed_size(M, K, "f16", n, m)
    vals, idx = dev_bytes(vb), dev_bytes(mb)
    nb.nm_compress(W.to(DEV), M, K, K, "f16", n, m, 0, nb.NM_META_CANONICAL, vals, idx)
    y = torch.empty((batch, M), dtype=torch.float16, device=DEV)
    plan = nb.nm_spmm_plan(nb.make_desc(M=M, N=batch, K=K, n=n, m=m, ab_type="f16", cd_type="f16", ldb=K, ldd=M,
                                        meta_layout=nb.NM_META_CANONICAL))
    nb.nm_spmm(plan, 1.0, vals, idx, x.to(DEV), 0.0, None, y)
    torch.cuda.synchronize()
    A = o.decode(o.nm_prune(inputs.as_numpy_bits(W), "f16", n, m)[0], "f16")
    ref = o.spmm(1.0, A, o.decode(inputs.as_numpy_bits(x), "f16").T)
    assert_gemm_close(y.cpu().double().numpy().T, ref, f"gather M={M} b={batch}")


def test_gather_ragged_and_beta():
    M, K, N, n, m = 77, 96, 11, 3, 8
    W = inputs.normal((M, K), 0.5, 9, "bf16")
    B = inputs.normal((N, K), 1.0, 10, "bf16")
    C = inputs.normal((M, N), 1.0, 11, "bf16")
    vb, mb = nb.nm_compressed_size(M, K, "bf16", n, m)
    vals, idx = dev_bytes(vb), dev_bytes(mb)
    nb.nm_compress(W.to(DEV), M, K, K, "bf16", n, m, 0, nb.NM_META_CANONICAL, vals, idx)
    Cd = C.to(DEV)
    D = torch.empty((M, 16), dtype=torch.bfloat16, device=DEV)  # ldd = 16 (row-major M x N, padded)
    Cp = torch.zeros((M, 16), dtype=torch.bfloat16, device=DEV)
    Cp[:, :N] = Cd
    plan = nb.nm_spmm_plan(nb.make_desc(M=M, N=N, K=K, n=n, m=m, ab_type="bf16", cd_type="bf16", ldb=K, ldc=16,
                                        ldd=16, order_cd=nb.NM_ROW, meta_layout=nb.NM_META_CANONICAL))
    nb.nm_spmm(plan, 0.5, vals, idx, B.to(DEV), -2.0, Cp, D)
    torch.cuda.synchronize()
    A = o.decode(o.nm_prune(inputs.as_numpy_bits(W), "bf16", n, m)[0], "bf16")
    ref = o.spmm(0.5, A, o.decode(inputs.as_numpy_bits(B), "bf16").T, -2.0, C.double().numpy())
    assert_gemm_close(D.cpu().double().numpy()[:, :N], ref, "gather ragged")


def test_k_zero_gives_beta_c():
    M, N = 64, 48
    C = inputs.normal((N, M), 1.0, 3, "f16").to(DEV)
    D = torch.empty((N, M), dtype=torch.float16, device=DEV)
    plan = nb.nm_spmm_plan(nb.make_desc(M=M, N=N, K=0, ab_type="f16", cd_type="f16", ldb=8, ldc=M, ldd=M))
    nb.nm_spmm(plan, 1.0, None, None, None, 0.5, C, D)
    torch.cuda.synchronize()
    assert torch.equal(D, (C.float() * 0.5).half())


# one row block (single CTA), two row blocks on paired CTAs (the default), two on single CTAs
@pytest.mark.parametrize("M,algo", [(128, 0), (256, 0), (256, 2)])
def test_bounded_wait_reports_timeout_and_context_survives(M, algo):
    """A wait nothing completes gives up after its budget: NM_ERR_TIMEOUT, no hang, GPU still usable."""
    N, K = 128, 256
    W = inputs.normal((M, K), 0.5, 1, "f16").to(DEV)
    X = inputs.normal((N, K), 1.0, 2, "f16").to(DEV)
    vals, meta = compress_on_gpu(W, M, K, "f16")
    D = torch.zeros((N, M), dtype=torch.float16, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    desc = nb.make_desc(M=M, N=N, K=K, ab_type="f16", cd_type="f16", ldb=K, ldd=M, algo=algo)
    nb.nm_test_spmm_wait_timeout(desc, vals, meta, X, D, status, budget_cycles=1 << 22)
    torch.cuda.synchronize()
    assert int(status.item()) == nb.NM_ERR_TIMEOUT
    # the context is intact: a normal product still runs and is right
    status.zero_()
    plan = nb.nm_spmm_plan(desc)
    nb.nm_spmm(plan, 1.0, vals, meta, X, 0.0, None, D, d_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    A = o.decode(o.nm_prune(bits_of(W, "f16", (M, K)), "f16", 2, 4)[0], "f16")
    ref = o.spmm(1.0, A, o.decode(bits_of(X, "f16", (N, K)), "f16").T)
    assert_gemm_close(D.cpu().double().numpy().T, ref, "after timeout")


I8_CASES = [
    # M, N, K, alpha, beta, order_cd, sampled, kind
    (128, 64, 128, 1, 0, nb.NM_COL, False, "uniform"),
    (200, 136, 192, 3, -2, nb.NM_ROW, False, "uniform"),      # ragged M/N, K tail of one k-step, alpha/beta
    (64, 128, 4096, 1, 0, nb.NM_COL, False, "extreme"),       # |products| at the int8 limit over K = 4096
    (1024, 4096, 1024, 1, 0, nb.NM_COL, True, "uniform"),     # BERT-Large shapes
    (4096, 4096, 1024, 1, 0, nb.NM_COL, True, "uniform"),
    (1024, 4096, 4096, 1, 0, nb.NM_COL, True, "uniform"),
]


@pytest.mark.parametrize("M,N,K,alpha,beta,order_cd,sampled,kind", I8_CASES)
def test_sparse_int8_bit_exact(M, N, K, alpha, beta, order_cd, sampled, kind):
    if kind == "extreme":
        W = torch.where(torch.arange(M * K).reshape(M, K) % 3 == 0, -128, 127).to(torch.int8)
        X = torch.where(torch.arange(N * K).reshape(N, K) % 5 == 0, -128, 127).to(torch.int8)
    else:
        W = inputs.uniform_int8((M, K), inputs.SEED_W + M)
        X = inputs.uniform_int8((N, K), inputs.SEED_X + N)
    vb, mb = nb.nm_compressed_size(M, K, "i8", 2, 4, nb.NM_META_CANONICAL)
    vals, meta = dev_bytes(vb), dev_bytes(mb)
    nb.nm_compress(W.to(DEV), M, K, K, "i8", 2, 4, 0, nb.NM_META_CANONICAL, vals, meta)
    cd_shape = (M, N) if order_cd == nb.NM_ROW else (N, M)
    C = torch.randint(-2**31, 2**31 - 1, cd_shape, dtype=torch.int64).to(torch.int32) if beta else None
    D = torch.full(cd_shape, 7, dtype=torch.int32, device=DEV)
    plan = nb.nm_spmm_plan(nb.make_desc(M=M, N=N, K=K, ab_type="i8", cd_type="i32", ldb=K,
                                        ldc=cd_shape[1] if beta else 0, ldd=cd_shape[1], order_cd=order_cd,
                                        meta_layout=nb.NM_META_CANONICAL))
    nb.nm_spmm(plan, alpha, vals, meta, X.to(DEV), beta, C.to(DEV) if C is not None else None, D)
    torch.cuda.synchronize()
    A = o.nm_prune(W.numpy(), "i8", 2, 4)[0]
    rows = sample_rows(M, 64, seed=M + K) if sampled else np.arange(M)
    Cm = None
    if C is not None:
        Cm = C.numpy() if order_cd == nb.NM_ROW else C.numpy().T
        Cm = Cm[rows]
    ref = o.spmm_int(alpha, A[rows], X.numpy().T, beta, Cm)
    got = D.cpu().numpy()
    got = got if order_cd == nb.NM_ROW else got.T
    assert np.array_equal(got[rows], ref)


@pytest.mark.parametrize("mode", ["sparse", "dense", "dense_odd"])
def test_search_keeps_a_correct_algorithm(mode):
    """Plan-time search (cuSPARSELt blog: algorithm selection, auto-tuning) picks one of the two
    tensor-core kernels, and the plan then computes the product correctly."""
    if mode == "sparse":
        M, N, K = 768, 4096, 768
        W = inputs.normal((M, K), 0.02, 31, "bf16")
        X = inputs.normal((N, K), 1.0, 32, "bf16")
        vals, meta = compress_on_gpu(W.to(DEV), M, K, "bf16")
        D = torch.empty((N, M), dtype=torch.bfloat16, device=DEV)
        plan = nb.nm_spmm_plan(nb.make_desc(M=M, N=N, K=K, ab_type="bf16", cd_type="bf16", ldb=K, ldd=M))
        args = (1.0, vals, meta, X.to(DEV), 0.0, None, D)
        ws, wsb = None, 0
    else:
        # dense: 6 row blocks (paired and single, K splits near the plan's); dense_odd: 3 row
        # blocks (the single-CTA kernel, K splits only)
        M, N, K = (768, 768, 4096) if mode == "dense" else (384, 512, 8192)
        dY = inputs.normal((K, M), 1.0, 33, "bf16")
        X = inputs.normal((K, N), 1.0, 34, "bf16")
        _, mask_ref = o.nm_prune(inputs.as_numpy_bits(inputs.normal((M, N), 0.02, 35, "bf16")), "bf16", 2, 4)
        bits = torch.from_numpy(o.mask_to_bits(mask_ref).view(np.int32)).to(DEV)
        D = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
        plan = nb.nm_spmm_plan(nb.make_desc(M=M, N=N, K=K, mode=nb.NM_SPMM_DENSE_MASKED, ab_type="bf16",
                                            cd_type="bf16", order_a=nb.NM_COL, order_b=nb.NM_ROW, order_cd=nb.NM_ROW,
                                            lda=M, ldb=N, ldd=N, meta_layout=nb.NM_META_CANONICAL))
        wsb = nb.nm_spmm_plan_workspace(plan)
        ws = dev_bytes(wsb) if wsb else None
        args = (1.0, dY.to(DEV), bits, X.to(DEV), 0.0, None, D)
    chosen = nb.nm_spmm_search(plan, *args, workspace=ws, workspace_bytes=wsb, repeats=2)
    if mode == "dense_odd":
        assert chosen == nb.NM_ALGO_DEFAULT
    else:
        assert chosen in (nb.NM_ALGO_PAIRED, nb.NM_ALGO_SINGLE)
    # the K split it keeps fits in the workspace it was given
    assert nb.nm_spmm_plan_workspace(plan) <= wsb
    assert nb.nm_spmm_plan_launches(plan) in (1, 2)
    # searched once: a second call reports the same choice
    assert nb.nm_spmm_search(plan, *args, workspace=ws, workspace_bytes=wsb, repeats=2) == chosen
    D.fill_(float("nan"))
    nb.nm_spmm(plan, *args, workspace=ws, workspace_bytes=wsb)
    torch.cuda.synchronize()
    if mode == "sparse":
        A = o.decode(o.nm_prune(inputs.as_numpy_bits(W), "bf16", 2, 4)[0], "bf16")
        rows = sample_rows(M, 128, seed=5)
        ref = o.spmm(1.0, A[rows], o.decode(inputs.as_numpy_bits(X), "bf16").T)
        assert_gemm_close(D.cpu().double().numpy().T[rows], ref, f"searched sparse (algo {chosen})")
    else:
        rows = sample_rows(M, 128, seed=6)
        ref = o.masked_weight_grad(o.decode(inputs.as_numpy_bits(dY), "bf16")[:, rows],
                                   o.decode(inputs.as_numpy_bits(X), "bf16"), mask_ref[rows])
        assert_gemm_close(D.cpu().double().numpy()[rows], ref, f"searched dense (algo {chosen})")


def test_first_call_from_a_new_host_thread():
    """A thread that has made no CUDA call yet (a framework's worker thread) gets a correct product
    on its first call: the library binds the device's context before encoding tensor maps."""
    import threading

    M, N, K = 256, 512, 256
    W = inputs.normal((M, K), 0.05, 51, "f16").to(DEV)
    X = inputs.normal((N, K), 1.0, 52, "f16").to(DEV)
    vals, meta = compress_on_gpu(W, M, K, "f16")
    D = torch.full((N, M), float("nan"), dtype=torch.float16, device=DEV)
    plan = nb.nm_spmm_plan(nb.make_desc(M=M, N=N, K=K, ab_type="f16", cd_type="f16", ldb=K, ldd=M))
    torch.cuda.synchronize()
    errors = []

    def run():
        try:
            nb.nm_spmm(plan, 1.0, vals, meta, X, 0.0, None, D, stream=0)
        except Exception as e:  # reported below
            errors.append(e)

    t = threading.Thread(target=run)
    t.start()
    t.join()
    torch.cuda.synchronize()
    assert not errors, errors
    A = o.decode(o.nm_prune(bits_of(W, "f16", (M, K)), "f16", 2, 4)[0], "f16")
    ref = o.spmm(1.0, A, o.decode(bits_of(X, "f16", (N, K)), "f16").T)
    assert_gemm_close(D.cpu().double().numpy().T, ref, "first call from a new thread")


@pytest.mark.parametrize("M,N,K,alpha,beta,order_cd", [
    (128, 64, 128, 0.5, 0.0, nb.NM_COL),
    (200, 144, 192, 0.03125, 0.75, nb.NM_ROW),   # ragged, with C
    (1024, 4096, 1024, 0.01, 0.0, nb.NM_COL),    # BERT-shaped
])
def test_sparse_int8_output_bit_exact(M, N, K, alpha, beta, order_cd):
    """INT8 inputs and output (cuSPARSELt blog, key features) with this library's float scale and rounding."""
    W = inputs.uniform_int8((M, K), 61 + M)
    X = inputs.uniform_int8((N, K), 62 + N)
    vb, mb = nb.nm_compressed_size(M, K, "i8", 2, 4, nb.NM_META_CANONICAL)
    vals, meta = dev_bytes(vb), dev_bytes(mb)
    nb.nm_compress(W.to(DEV), M, K, K, "i8", 2, 4, 0, nb.NM_META_CANONICAL, vals, meta)
    cd_shape = (M, N) if order_cd == nb.NM_ROW else (N, M)
    ld = (cd_shape[1] + 15) // 16 * 16
    C = inputs.uniform_int8(cd_shape, 63) if beta else None
    Cp = None
    if C is not None:
        Cp = torch.zeros((cd_shape[0], ld), dtype=torch.int8)
        Cp[:, :cd_shape[1]] = C
        Cp = Cp.to(DEV)
    D = torch.full((cd_shape[0], ld), 99, dtype=torch.int8, device=DEV)
    plan = nb.nm_spmm_plan(nb.make_desc(M=M, N=N, K=K, ab_type="i8", cd_type="i8", ldb=K, ldc=ld if beta else 0,
                                        ldd=ld, order_cd=order_cd, meta_layout=nb.NM_META_CANONICAL))
    nb.nm_spmm(plan, alpha, vals, meta, X.to(DEV), beta, Cp, D)
    torch.cuda.synchronize()
    A = o.nm_prune(W.numpy(), "i8", 2, 4)[0]
    Cm = None
    if C is not None:
        Cm = C.numpy() if order_cd == nb.NM_ROW else C.numpy().T
    ref = o.spmm_int8_out(alpha, A, X.numpy().T, beta, Cm)
    got = D.cpu().numpy()[:, :cd_shape[1]]
    got = got if order_cd == nb.NM_ROW else got.T
    assert np.array_equal(got, ref)


def test_i8_sparse_mma_rate_probe():
    """The measurement hook behind the int8 rows' roofline fraction returns a plausible rate."""
    peak = nb.nm_test_i8_sparse_mma_rate(2000)
    assert 10.0 < peak < 5000.0
    with pytest.raises(nb.NmError):
        nb.nm_test_i8_sparse_mma_rate(0)


def test_masked_weight_grad_fused_splits_workspace():
    """Two K splits summed in the paired product: a workspace of garbage works, its arrival
    words (the last tiles x 8 warps x 8 bytes) are 0 after the call, and a second call on the
    same workspace gives the same D."""
    M, N, K, dtype = 3072, 768, 16384, "bf16"
    dY = inputs.normal((K, M), 1.0, inputs.SEED_DY + K, dtype)
    X = inputs.normal((K, N), 1.0, inputs.SEED_X + K, dtype)
    W = inputs.normal((M, N), 0.02, inputs.SEED_W, dtype)
    _, mask_ref = o.nm_prune(inputs.as_numpy_bits(W), dtype, 2, 4)
    bits = torch.from_numpy(o.mask_to_bits(mask_ref).view(np.int32)).to(DEV)
    plan = nb.nm_spmm_plan(nb.make_desc(M=M, N=N, K=K, mode=nb.NM_SPMM_DENSE_MASKED, ab_type=dtype, cd_type=dtype,
                                        order_a=nb.NM_COL, order_b=nb.NM_ROW, order_cd=nb.NM_ROW, lda=M, ldb=N,
                                        ldd=N, meta_layout=nb.NM_META_CANONICAL))
    assert nb.nm_spmm_plan_launches(plan) == 1
    ws_bytes = nb.nm_spmm_plan_workspace(plan)
    ws = torch.full((ws_bytes,), 0xA5, dtype=torch.uint8, device=DEV)
    words = ((M + 127) // 128) * ((N + 255) // 256) * 8 * 8
    dYd, Xd = dY.to(DEV), X.to(DEV)
    outs = []
    for _ in range(2):
        dW = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=DEV)
        nb.nm_spmm(plan, 1.0, dYd, bits, Xd, 0.0, None, dW, ws, ws_bytes)
        torch.cuda.synchronize()
        assert int(ws[ws_bytes - words:].count_nonzero().item()) == 0
        outs.append(dW.view(torch.int16).clone())
    assert torch.equal(outs[0], outs[1])
    rows = sample_rows(M, 64, seed=5)
    ref = o.masked_weight_grad(o.decode(inputs.as_numpy_bits(dY), dtype)[:, rows],
                               o.decode(inputs.as_numpy_bits(X), dtype), mask_ref[rows])
    got = outs[0].view(torch.bfloat16).cpu().double().numpy()[rows]
    assert_gemm_close(got, ref, "fused dW")
