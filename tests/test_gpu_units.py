"""GPU parity of vector-wise (1 x 32) and block-wise (32 x 32) pruning and of
the product over the kept units, against the CPU oracle.  Masks, CSR arrays,
packed values and pruned copies are compared bit for bit; products within the
FP16/BF16 tolerance."""
import numpy as np
import pytest
import torch

import oracle as o
from structured_sparse_gemm_nm_gb300 import binding as nb
from structured_sparse_gemm_nm_gb300 import inputs

from gpu_util import DEV, ESIZE, assert_gemm_close, bits_of, dev_bytes, ensure_lib, to_dev_bits, u32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_lib()


def host_matrix(rows, cols, dtype, seed, kind):
    rng = np.random.default_rng(seed)
    if dtype == "i8":
        if kind == "ties":
            return rng.integers(-2, 3, size=(rows, cols)).astype(np.int8)
        return inputs.as_numpy_bits(inputs.uniform_int8((rows, cols), seed, -128, 127))
    if kind == "zeros":
        return np.zeros((rows, cols), np.uint16)
    if kind == "ties":  # small integers: many units share a score
        return rng.integers(-2, 3, size=(rows, cols)).astype(np.float16).view(np.uint16)
    a = inputs.as_numpy_bits(inputs.normal((rows, cols), 0.02, seed, "f16")).copy()
    if kind == "special":
        pool = np.array([0.0, -0.0, 1.0, -1.0, np.inf, -np.inf, np.nan], np.float16).view(np.uint16)
        idx = rng.choice(a.size, size=max(1, a.size // 200), replace=False)
        a.reshape(-1)[idx] = rng.choice(pool, size=idx.size)
    if kind == "mixed":  # every finite exponent (subnormals to 65504) with random signs
        bits = rng.integers(0, 0x7C00, size=(rows, cols)) | (rng.integers(0, 2, size=(rows, cols)) << 15)
        return bits.astype(np.uint16)
    if kind == "large":  # magnitudes near the top of the f16 range: the widest exact scores
        a = (rng.uniform(30000, 65504, size=(rows, cols)) * rng.choice([-1, 1], size=(rows, cols)))
        a = a.astype(np.float16).view(np.uint16)
    return a


def run_units(W, rows, cols, dtype, bh, keep, score="abs_of_sum", ld=None, in_place=False):
    """Runs the GPU pruning; returns host copies of every output."""
    ld = ld or cols
    es = ESIZE[dtype]
    pad = np.zeros((rows, ld), W.dtype)
    pad[:, :cols] = W
    if ld > cols:
        pad[:, cols:] = 0x3C00 if dtype != "i8" else 7
    Wd = to_dev_bits(pad, dtype)
    units = (rows // bh) * (cols // 32)
    urows = rows // bh
    Wo = Wd if in_place else dev_bytes(rows * ld * es, fill=0xAB)
    mask = dev_bytes(rows * (cols // 32) * 4, fill=0xCD)
    csr = dev_bytes((urows + 1 + keep) * 4, fill=0xEF)
    vals = dev_bytes(max(1, keep) * bh * 32 * es, fill=0x5A)
    wsb = nb.nm_prune_units_workspace(rows, cols, bh, 32)
    ws = dev_bytes(wsb, fill=0x77)  # contents must not matter
    if bh == 1:
        nb.nm_prune_vector_wise(Wd, rows, cols, ld, dtype, 32, keep,
                                nb.NM_SCORE_ABS_OF_SUM if score == "abs_of_sum" else nb.NM_SCORE_SUM_OF_ABS,
                                W_out=Wo, ld_out=ld, mask_bits=mask, csr=csr, vals=vals, workspace=ws,
                                workspace_bytes=wsb)
    else:
        nb.nm_prune_block_wise(Wd, rows, cols, ld, dtype, bh, 32, keep, W_out=Wo, ld_out=ld, mask_bits=mask,
                               csr=csr, vals=vals, workspace=ws, workspace_bytes=wsb)
    torch.cuda.synchronize()
    got_w = bits_of(Wo, dtype, (rows, ld))
    return dict(W_out=got_w, in_place=in_place, mask=u32(mask, rows * (cols // 32)).reshape(rows, cols // 32),
                csr=u32(csr, urows + 1 + keep).view(np.int32),
                vals=bits_of(vals, dtype, (keep * bh * 32,)) if keep else np.zeros(0, W.dtype), pad=pad, units=units)


def check_against_oracle(W, rows, cols, dtype, bh, density, score, got, ld):
    units = got["units"]
    if bh == 1:
        mask = o.vector_wise_mask(W, dtype, density, 32, score)
        csr, vals = o.vector_wise_csr(W, mask, 32)
    else:
        mask = o.block_wise_mask(W, dtype, density, 32, 32)
        csr, vals = o.block_wise_csr(W, mask, 32, 32)
    keep = int(units * density)
    assert int(mask.sum()) == keep * bh * 32
    assert (got["mask"] == o.mask_to_bits(mask)).all(), "mask bits"
    assert (got["csr"] == csr).all(), "csr"
    assert (got["vals"] == vals.reshape(-1)).all(), "vals"
    assert (got["W_out"][:, :cols] == np.where(mask, W, 0)).all(), "pruned copy"
    if ld > cols:  # the columns past `cols` keep what was there: W's padding in place, else the 0xAB fill
        if got["in_place"]:
            before = got["pad"][:, cols:]
        else:
            before = np.full((rows, ld - cols), 0xAB, np.uint8).view(np.int8) if dtype == "i8" else \
                np.full((rows, ld - cols), 0xABAB, np.uint16)
        assert (got["W_out"][:, cols:] == before).all(), "padding touched"


UNIT_CASES = [
    # rows, cols, ld, dtype, bh, density, score, kind
    (64, 128, 128, "f16", 1, 0.25, "abs_of_sum", "normal"),
    (100, 96, 104, "f16", 1, 0.3, "abs_of_sum", "special"),
    (100, 96, 96, "f16", 1, 0.3, "sum_of_abs", "special"),
    (33, 256, 256, "i8", 1, 0.5, "abs_of_sum", "normal"),
    (33, 256, 272, "i8", 1, 0.5, "sum_of_abs", "ties"),
    (257, 64, 64, "f16", 1, 0.4, "abs_of_sum", "ties"),
    (2048, 2048, 2048, "f16", 1, 0.3, "abs_of_sum", "ties"),  # thousands of keys in the threshold bucket
    (128, 128, 128, "f16", 1, 0.5, "abs_of_sum", "zeros"),
    (64, 256, 256, "f16", 1, 0.25, "sum_of_abs", "large"),
    (64, 256, 256, "f16", 1, 0.25, "abs_of_sum", "large"),
    (96, 512, 512, "f16", 1, 0.3, "abs_of_sum", "mixed"),
    (96, 512, 512, "f16", 1, 0.3, "sum_of_abs", "mixed"),
    (128, 256, 256, "f16", 32, 0.4, "sum_of_abs", "mixed"),
    (64, 64, 64, "f16", 1, 0.0, "abs_of_sum", "normal"),
    (64, 64, 64, "f16", 1, 1.0, "abs_of_sum", "normal"),
    (1, 32, 32, "f16", 1, 1.0, "abs_of_sum", "normal"),
    (4096, 4096, 4096, "f16", 1, 0.25, "abs_of_sum", "normal"),
    (64, 96, 96, "f16", 32, 0.25, "sum_of_abs", "normal"),
    (96, 128, 136, "f16", 32, 0.5, "sum_of_abs", "special"),
    (64, 64, 64, "i8", 32, 0.5, "sum_of_abs", "normal"),
    (256, 288, 288, "f16", 32, 0.3, "sum_of_abs", "ties"),
    (128, 128, 128, "f16", 32, 0.5, "sum_of_abs", "large"),
    (64, 64, 64, "f16", 32, 0.0, "sum_of_abs", "normal"),
    (64, 64, 64, "f16", 32, 1.0, "sum_of_abs", "normal"),
    (4096, 4096, 4096, "f16", 32, 0.25, "sum_of_abs", "normal"),
]


@pytest.mark.parametrize("rows,cols,ld,dtype,bh,density,score,kind", UNIT_CASES)
def test_unit_pruning_matches_oracle(rows, cols, ld, dtype, bh, density, score, kind):
    W = host_matrix(rows, cols, dtype, 50 + rows + cols + bh, kind)
    units = (rows // bh) * (cols // 32)
    keep = int(units * density)
    got = run_units(W, rows, cols, dtype, bh, keep, score, ld=ld)
    check_against_oracle(W, rows, cols, dtype, bh, density, score, got, ld)


def test_unit_pruning_one_crowded_bucket():
    # 2.6 M vectors whose scores all fall in one histogram bucket (1.0 everywhere, a tenth
    # of the elements one ulp higher: 15 distinct scores): every candidates CTA holds
    # more keys than its shared buffer, the radix search runs over millions of keys in
    # global memory, and thousands of units tie at the threshold
    rows, cols = 5120, 16384
    rng = np.random.default_rng(7)
    W = np.full((rows, cols), 0x3C00, np.uint16)
    W[rng.random((rows, cols)) < 0.1] = 0x3C01
    keep = int(rows * cols // 32 * 0.3)
    got = run_units(W, rows, cols, "f16", 1, keep, "abs_of_sum")
    check_against_oracle(W, rows, cols, "f16", 1, 0.3, "abs_of_sum", got, cols)


def test_unit_pruning_in_place_and_repeatable():
    rows, cols = 96, 160
    W = host_matrix(rows, cols, "f16", 61, "normal")
    keep = int(rows * cols // 32 * 0.25)
    first = run_units(W, rows, cols, "f16", 1, keep, in_place=False)
    again = run_units(W, rows, cols, "f16", 1, keep, in_place=True)
    for k in ("mask", "csr", "vals", "W_out"):
        assert (first[k] == again[k]).all(), k
    check_against_oracle(W, rows, cols, "f16", 1, 0.25, "abs_of_sum", again, cols)


# ------------------------------------------------------------------ product
def unit_product(vals_bits, csr, M, K, N, dtype, bh, B_bits, alpha=1.0, beta=0.0, C_bits=None, order_cd=nb.NM_ROW,
                 ldb=None):
    ldb = ldb or K
    ldd = N if order_cd == nb.NM_ROW else M
    desc = nb.make_desc(M=M, N=N, K=K, mode=nb.NM_SPMM_BLOCK_SPARSE_A, n=bh, m=32, ab_type=dtype, cd_type=dtype,
                        order_b=nb.NM_COL, order_cd=order_cd, ldb=ldb, ldc=ldd if C_bits is not None else 0,
                        ldd=ldd, meta_layout=nb.NM_META_CANONICAL)
    plan = nb.nm_spmm_plan(desc)
    A = to_dev_bits(vals_bits.reshape(-1) if vals_bits.size else np.zeros(8, vals_bits.dtype), dtype)
    meta = torch.from_numpy(np.ascontiguousarray(csr.astype(np.int32))).to(DEV)
    Bp = np.zeros((N, ldb), np.uint16)
    Bp[:, :K] = B_bits
    Bd = to_dev_bits(Bp, dtype)
    shape = (M, N) if order_cd == nb.NM_ROW else (N, M)
    D = dev_bytes(M * N * 2, fill=0x7E)
    Cd = to_dev_bits(C_bits, dtype) if C_bits is not None else None
    nb.nm_spmm(plan, alpha, A, meta, Bd, beta, Cd, D)
    torch.cuda.synchronize()
    plan.destroy()
    return o.decode(bits_of(D, dtype, shape), dtype)


PRODUCT_CASES = [
    # rows, cols, bh, N, dtype, alpha, beta, order_cd
    (64, 128, 1, 1, "f16", 1.0, 0.0, nb.NM_ROW),
    (64, 128, 1, 8, "f16", 1.0, 0.0, nb.NM_ROW),
    (96, 256, 1, 5, "bf16", 0.5, -1.0, nb.NM_COL),
    (96, 256, 1, 11, "f16", 1.0, 0.25, nb.NM_ROW),
    (64, 128, 32, 1, "f16", 1.0, 0.0, nb.NM_ROW),
    (128, 256, 32, 8, "bf16", 1.0, 0.0, nb.NM_COL),
    (96, 96, 32, 13, "f16", 2.0, 0.5, nb.NM_ROW),
    (12000, 64, 1, 1, "f16", 1.0, 0.0, nb.NM_ROW),  # several interleaved rows per warp
    (12000, 64, 1, 8, "f16", 1.0, 0.0, nb.NM_COL),
    (4096, 4096, 1, 1, "f16", 1.0, 0.0, nb.NM_ROW),
    (4096, 4096, 1, 8, "f16", 1.0, 0.0, nb.NM_ROW),
    (4096, 4096, 32, 1, "f16", 1.0, 0.0, nb.NM_ROW),
    (4096, 4096, 32, 8, "f16", 1.0, 0.0, nb.NM_ROW),
]


@pytest.mark.parametrize("rows,cols,bh,N,dtype,alpha,beta,order_cd", PRODUCT_CASES)
def test_unit_product_matches_oracle(rows, cols, bh, N, dtype, alpha, beta, order_cd):
    seed = 70 + rows + N + bh
    W = inputs.as_numpy_bits(inputs.normal((rows, cols), 0.02, seed, "f16"))
    # the selection is defined on f16 scores; a bf16 product reuses the same pattern on bf16 values
    if bh == 1:
        mask = o.vector_wise_mask(W, "f16", 0.25, 32)
    else:
        mask = o.block_wise_mask(W, "f16", 0.25, 32, 32)
    Wt = W if dtype == "f16" else inputs.as_numpy_bits(inputs.normal((rows, cols), 0.02, seed, "bf16"))
    csr, vals = (o.vector_wise_csr(Wt, mask, 32) if bh == 1 else o.block_wise_csr(Wt, mask, 32, 32))
    B = inputs.as_numpy_bits(inputs.normal((N, cols), 1.0, seed + 1, dtype))
    C = None
    if beta != 0.0:
        shape = (rows, N) if order_cd == nb.NM_ROW else (N, rows)
        C = inputs.as_numpy_bits(inputs.normal(shape, 1.0, seed + 2, dtype))
    got = unit_product(vals, csr, rows, cols, N, dtype, bh, B, alpha, beta, C, order_cd)
    A = o.decode(np.where(mask, Wt, 0), dtype)
    Cref = None
    if C is not None:
        Cref = o.decode(C, dtype) if order_cd == nb.NM_ROW else o.decode(C, dtype).T
    ref = o.spmm(alpha, A, o.decode(B, dtype).T, beta, Cref)
    if order_cd == nb.NM_COL:
        got = got.T
    assert_gemm_close(got, ref, f"unit product {rows}x{cols} bh={bh} N={N}")


def test_unit_product_from_gpu_pruning():
    """The product consumes what the pruning wrote, end to end on the device."""
    rows, cols, N = 256, 512, 8
    W = host_matrix(rows, cols, "f16", 81, "normal")
    keep = int(rows * cols // 32 * 0.25)
    got = run_units(W, rows, cols, "f16", 1, keep)
    B = inputs.as_numpy_bits(inputs.normal((N, cols), 1.0, 82, "f16"))
    D = unit_product(got["vals"], got["csr"], rows, cols, N, "f16", 1, B)
    mask = o.vector_wise_mask(W, "f16", 0.25, 32)
    ref = o.spmm(1.0, o.decode(np.where(mask, W, 0), "f16"), o.decode(B, "f16").T)
    assert_gemm_close(D, ref, "pruning -> product")
