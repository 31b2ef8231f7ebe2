"""Host-side checks of the C ABI: the library loads, exports every declared
entry point, and rejects bad arguments before touching CUDA."""
import ctypes
import os
import re
import subprocess

import pytest

from structured_sparse_gemm_nm_gb300 import binding as nb

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "nm.h")
TESTING_HEADER = os.path.join(ROOT, "include", "nm_testing.h")


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(nb.LIB_PATH):
        from structured_sparse_gemm_nm_gb300.build import build

        build()
    return nb.lib()


def declared_functions(header=HEADER):
    text = open(header).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(nm_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_binding_names():
    assert declared_functions() == sorted(nb.EXPORTED)
    assert declared_functions(TESTING_HEADER) == sorted(nb.TESTING_EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", nb.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r" T (nm_[a-z0-9_]+)", out))
    declared = declared_functions() + declared_functions(TESTING_HEADER)
    missing = [f for f in declared if f not in exported]
    assert not missing, missing
    # nothing is exported that a header does not declare
    assert exported == set(declared), sorted(exported - set(declared))
    for f in declared:
        assert hasattr(lib, f)


def test_version_and_status_strings(lib):
    assert nb.nm_version() == 1
    for code, name in enumerate(["NM_OK", "NM_ERR_INVALID_ARG", "NM_ERR_UNSUPPORTED", "NM_ERR_MISALIGNED",
                                 "NM_ERR_CUDA", "NM_ERR_TIMEOUT"]):
        assert nb.status_string(code) == name


def test_compressed_size(lib):
    assert nb.nm_compressed_size(64, 128, "f16", 2, 4) == (64 * 64 * 2, 64 * 8 * 2)
    # tensor-core order: slot rows padded to 128, one word per slot and k-step
    assert nb.nm_compressed_size(64, 128, "f16", 2, 4, nb.NM_META_TC) == (64 * 64 * 2, 4 * 128 * 4)
    assert nb.nm_compressed_size(300, 96, "bf16", 2, 4, nb.NM_META_TC) == (300 * 48 * 2, 3 * 384 * 4)
    assert nb.nm_compressed_size(4096, 4096, "f16", 8, 32) == (4096 * 1024 * 2, 4096 * 1024)
    assert nb.nm_compressed_size(8, 64, "i8", 2, 4) == (8 * 32, 8 * 4 * 2)
    assert nb.nm_compressed_size(8, 20, "f16", 2, 4)[1] == 8 * 2 * 2  # ceil(20/16) words per row
    with pytest.raises(nb.NmError) as e:
        nb.nm_compressed_size(8, 64, "i8", 2, 4, nb.NM_META_TC)
    assert e.value.status == nb.NM_ERR_UNSUPPORTED
    with pytest.raises(nb.NmError):
        nb.nm_compressed_size(8, 48, "f16", 2, 4, nb.NM_META_TC)  # cols % 32
    with pytest.raises(nb.NmError):
        nb.nm_compressed_size(8, 64, "f16", 4, 32, nb.NM_META_TC)


FAKE = 0x10000  # never dereferenced: every call below fails validation first


@pytest.mark.parametrize(
    "kwargs,status",
    [
        (dict(n=4, m=4), nb.NM_ERR_INVALID_ARG),
        (dict(n=0, m=4), nb.NM_ERR_INVALID_ARG),
        (dict(n=2, m=33), nb.NM_ERR_INVALID_ARG),
        (dict(cols=30), nb.NM_ERR_INVALID_ARG),
        (dict(ld=10), nb.NM_ERR_INVALID_ARG),
        (dict(W=None), nb.NM_ERR_INVALID_ARG),
        (dict(W=FAKE + 1), nb.NM_ERR_MISALIGNED),
        (dict(dtype=nb.NM_F32), nb.NM_ERR_INVALID_ARG),
        (dict(W_out=FAKE, ld_out=64), nb.NM_ERR_INVALID_ARG),  # aliasing W with another ld
    ],
)
def test_prune_rejects_bad_arguments(lib, kwargs, status):
    a = dict(W=FAKE, rows=8, cols=32, ld=32, dtype=nb.NM_F16, n=2, m=4, W_out=None, ld_out=0, mask_bits=None)
    a.update(kwargs)
    st = lib.nm_prune(a["W"], a["rows"], a["cols"], a["ld"], a["dtype"], a["n"], a["m"], a["W_out"], a["ld_out"],
                      a["mask_bits"], None)
    assert st == status


def test_other_calls_reject_bad_arguments(lib):
    L = lib
    assert L.nm_compress(FAKE, 8, 32, 32, nb.NM_F16, 2, 4, 2, 0, None, None, None) == nb.NM_ERR_INVALID_ARG
    assert L.nm_compress(FAKE, 8, 48, 48, nb.NM_F16, 2, 4, 0, nb.NM_META_TC, None, None, None) == nb.NM_ERR_UNSUPPORTED
    assert L.nm_compress(FAKE, 8, 32, 32, nb.NM_F16, 2, 4, 0, 0, FAKE + 1, None, None) == nb.NM_ERR_MISALIGNED
    assert L.nm_decompress(None, None, 8, 32, nb.NM_F16, 2, 4, 0, FAKE, 32, None) == nb.NM_ERR_INVALID_ARG
    assert L.nm_check(FAKE, 8, 32, 32, nb.NM_F16, 2, 4, 0, None, None) == nb.NM_ERR_INVALID_ARG
    assert L.nm_check(FAKE, 6, 32, 32, nb.NM_F16, 2, 4, 1, FAKE, None) == nb.NM_ERR_INVALID_ARG  # rows % 4
    assert L.nm_check(FAKE, 8, 32, 32, nb.NM_F16, 8, 32, 1, FAKE, None) == nb.NM_ERR_INVALID_ARG  # not 2:4
    assert (L.nm_prune_transposable(FAKE, 6, 32, 32, nb.NM_F16, None, 0, None, None, None, None, None, 0, None)
            == nb.NM_ERR_INVALID_ARG)
    assert (L.nm_prune_transposable(FAKE, 8, 48, 48, nb.NM_F16, None, 0, None, None, FAKE, None, None, nb.NM_META_TC,
                                    None) == nb.NM_ERR_UNSUPPORTED)


def test_unit_pruning_rejects_bad_arguments(lib):
    L = lib
    ws = ctypes.c_size_t()
    assert L.nm_prune_units_workspace(64, 128, 1, 32, ctypes.byref(ws)) == nb.NM_OK and ws.value > 256 * 8
    assert L.nm_prune_units_workspace(64, 128, 1, 16, ctypes.byref(ws)) == nb.NM_ERR_UNSUPPORTED
    assert L.nm_prune_units_workspace(48, 128, 32, 32, ctypes.byref(ws)) == nb.NM_ERR_INVALID_ARG  # rows % 32
    assert L.nm_prune_units_workspace(0, 128, 1, 32, ctypes.byref(ws)) == nb.NM_OK and ws.value == 0
    big = 1 << 40

    def vw(**kw):
        a = dict(W=FAKE, rows=64, cols=128, ld=128, dt=nb.NM_F16, v=32, keep=64, score=0, W_out=None, ld_out=0,
                 mask=None, csr=FAKE, vals=None, ws=FAKE, wsb=big)
        a.update(kw)
        return L.nm_prune_vector_wise(a["W"], a["rows"], a["cols"], a["ld"], a["dt"], a["v"], a["keep"], a["score"],
                                      a["W_out"], a["ld_out"], a["mask"], a["csr"], a["vals"], a["ws"], a["wsb"],
                                      None)

    assert vw(dt=nb.NM_BF16) == nb.NM_ERR_UNSUPPORTED  # scores would not be exact
    assert vw(v=64) == nb.NM_ERR_UNSUPPORTED
    assert vw(cols=112, ld=112) == nb.NM_ERR_INVALID_ARG
    assert vw(keep=257) == nb.NM_ERR_INVALID_ARG
    assert vw(keep=-1) == nb.NM_ERR_INVALID_ARG
    assert vw(score=2) == nb.NM_ERR_INVALID_ARG
    assert vw(wsb=16) == nb.NM_ERR_INVALID_ARG
    assert vw(ws=None) == nb.NM_ERR_INVALID_ARG
    assert vw(ld=132) == nb.NM_ERR_MISALIGNED
    assert vw(vals=FAKE + 4) == nb.NM_ERR_MISALIGNED
    assert vw(W_out=FAKE, ld_out=136) == nb.NM_ERR_INVALID_ARG  # aliases W with another ld
    assert (L.nm_prune_block_wise(FAKE, 64, 128, 128, nb.NM_F16, 1, 32, 1, None, 0, None, None, None, FAKE, big, None)
            == nb.NM_ERR_UNSUPPORTED)
    assert (L.nm_prune_block_wise(FAKE, 64, 128, 128, nb.NM_I8, 32, 32, 9, None, 0, None, None, None, FAKE, big, None)
            == nb.NM_ERR_INVALID_ARG)  # 8 blocks


def plan_status(**kw):
    d = nb.make_desc(**kw)
    h = ctypes.c_void_p()
    st = nb.lib().nm_spmm_plan(ctypes.byref(h), ctypes.byref(d))
    if st == nb.NM_OK:
        nb.lib().nm_spmm_plan_destroy(h)
    return st


def test_plan_validation(lib):
    base = dict(M=256, N=512, K=1024, ab_type="f16", cd_type="f16", ldb=1024, ldd=256)
    assert plan_status(**base) == nb.NM_OK
    assert plan_status(**{**base, "cd_type": "bf16"}) == nb.NM_ERR_UNSUPPORTED
    assert plan_status(**{**base, "order_b": nb.NM_ROW, "ldb": 512}) == nb.NM_ERR_UNSUPPORTED
    assert plan_status(**{**base, "meta_layout": nb.NM_META_CANONICAL}) == nb.NM_ERR_UNSUPPORTED
    assert plan_status(**{**base, "ldb": 1000}) == nb.NM_ERR_INVALID_ARG  # < K
    assert plan_status(**{**base, "ldb": 1028}) == nb.NM_ERR_MISALIGNED   # not 16 bytes
    assert plan_status(**{**base, "K": 1000, "ldb": 1024}) == nb.NM_ERR_UNSUPPORTED  # K % 32
    assert plan_status(**{**base, "n": 8, "m": 32, "meta_layout": nb.NM_META_CANONICAL}) == nb.NM_OK
    dense = dict(M=256, N=512, K=4096, mode=nb.NM_SPMM_DENSE_MASKED, ab_type="bf16", cd_type="bf16",
                 order_a=nb.NM_COL, order_b=nb.NM_ROW, order_cd=nb.NM_ROW, lda=256, ldb=512, ldd=512)
    assert plan_status(**dense) == nb.NM_OK
    assert plan_status(**{**dense, "lda": 100}) == nb.NM_ERR_INVALID_ARG
    assert plan_status(**{**dense, "mode": 7}) == nb.NM_ERR_INVALID_ARG
    assert plan_status(M=-1, N=1, K=32, ab_type="f16", cd_type="f16", ldb=32, ldd=8) == nb.NM_ERR_INVALID_ARG
    assert plan_status(**{**base, "algo": nb.NM_ALGO_PAIRED}) == nb.NM_OK
    assert plan_status(**{**base, "algo": nb.NM_ALGO_SINGLE}) == nb.NM_OK
    assert plan_status(**{**base, "algo": 3}) == nb.NM_ERR_INVALID_ARG
    # fp32 C/D from 16-bit inputs on the tensor-core products only
    assert plan_status(**{**base, "cd_type": "f32"}) == nb.NM_OK
    assert plan_status(**{**base, "cd_type": "f32", "ldd": 258}) == nb.NM_ERR_MISALIGNED  # 1032 bytes
    assert plan_status(**{**dense, "cd_type": "f32"}) == nb.NM_OK
    assert plan_status(**{**base, "n": 8, "m": 32, "meta_layout": nb.NM_META_CANONICAL,
                          "cd_type": "f32"}) == nb.NM_ERR_UNSUPPORTED
    assert plan_status(**{**base, "ab_type": "i8", "cd_type": "f32",
                          "meta_layout": nb.NM_META_CANONICAL}) == nb.NM_ERR_UNSUPPORTED
    # an int8 output on the int8 sparse product only
    assert plan_status(**{**base, "ab_type": "i8", "cd_type": "i8", "meta_layout": nb.NM_META_CANONICAL}) == nb.NM_OK
    assert plan_status(**{**base, "ab_type": "i8", "cd_type": "i8", "n": 8, "m": 32,
                          "meta_layout": nb.NM_META_CANONICAL}) == nb.NM_ERR_UNSUPPORTED
    units = dict(M=256, N=8, K=1024, mode=nb.NM_SPMM_BLOCK_SPARSE_A, n=1, m=32, ab_type="f16", cd_type="f16",
                 ldb=1024, ldd=256)
    assert plan_status(**units) == nb.NM_OK
    assert plan_status(**{**units, "n": 32}) == nb.NM_OK
    assert plan_status(**{**units, "n": 16}) == nb.NM_ERR_UNSUPPORTED
    assert plan_status(**{**units, "n": 32, "M": 240}) == nb.NM_ERR_INVALID_ARG
    assert plan_status(**{**units, "ab_type": "i8", "cd_type": "i32"}) == nb.NM_ERR_UNSUPPORTED


def test_spmm_rejects_bad_pointers(lib):
    plan = nb.nm_spmm_plan(nb.make_desc(M=128, N=128, K=128, ab_type="f16", cd_type="f16", ldb=128, ldd=128))
    with pytest.raises(nb.NmError) as e:
        nb.nm_spmm(plan, 1.0, FAKE, FAKE, FAKE, 1.0, None, FAKE, stream=0)  # beta != 0 without C
    assert e.value.status == nb.NM_ERR_INVALID_ARG
    with pytest.raises(nb.NmError) as e:
        nb.nm_spmm(plan, 1.0, FAKE + 8, FAKE, FAKE, 0.0, None, FAKE, stream=0)
    assert e.value.status == nb.NM_ERR_MISALIGNED
    plan.destroy()


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(nb, "LIB_PATH", str(tmp_path / "absent.so"))
    monkeypatch.setattr(nb, "_lib", None)
    with pytest.raises(RuntimeError, match="no fallback"):
        nb.lib()


def test_noalloc_limit_matches_header():
    text = open(HEADER).read()
    m = re.search(r"#define NM_NOALLOC_MAX_UNITS (\d+)", text)
    assert m and int(m.group(1)) == nb.NM_NOALLOC_MAX_UNITS


def test_noalloc_rejects_bad_arguments_before_any_cuda_call(lib):
    # on a machine without a GPU these return their status without touching CUDA
    L = nb.lib()
    args = dict(rows=64, cols=128, ld=128, dtype=nb.NM_F16, v=32, keep=4, score=nb.NM_SCORE_ABS_OF_SUM)

    def call(W=FAKE, W_out=None, ld_out=0, mask=None, csr=None, vals=None, **kw):
        a = {**args, **kw}
        return L.nm_prune_vector_wise_noalloc(W, a["rows"], a["cols"], a["ld"], a["dtype"], a["v"], a["keep"],
                                              a["score"], W_out, ld_out, mask, csr, vals, None)

    assert call(W=FAKE + 8) == nb.NM_ERR_MISALIGNED          # W not 16-byte aligned
    assert call(ld=132) == nb.NM_ERR_MISALIGNED               # row pitch not a multiple of 16 bytes
    assert call(vals=FAKE + 4) == nb.NM_ERR_MISALIGNED
    assert call(csr=FAKE + 2) == nb.NM_ERR_MISALIGNED
    assert call(W_out=FAKE, ld_out=136) == nb.NM_ERR_INVALID_ARG  # aliases W with another ld
    assert call(keep=10**6) == nb.NM_ERR_INVALID_ARG
    assert call(dtype=nb.NM_BF16) == nb.NM_ERR_UNSUPPORTED
    assert call(v=16) == nb.NM_ERR_UNSUPPORTED
    assert call(rows=4096, cols=4128, ld=4128) == nb.NM_ERR_UNSUPPORTED  # beyond the fixed scratch


def test_i8_rate_probe_rejects_bad_arguments_before_any_cuda_call(lib):
    import ctypes
    L = nb.lib()
    ms, ops = ctypes.c_float(), ctypes.c_double()
    assert L.nm_test_i8_sparse_mma_rate(0, ctypes.byref(ms), ctypes.byref(ops)) == nb.NM_ERR_INVALID_ARG
    assert L.nm_test_i8_sparse_mma_rate(10**7, ctypes.byref(ms), ctypes.byref(ops)) == nb.NM_ERR_INVALID_ARG
    assert L.nm_test_i8_sparse_mma_rate(100, None, ctypes.byref(ops)) == nb.NM_ERR_INVALID_ARG


def test_search_argument_checks_and_fixed_plans(lib):
    plan = nb.nm_spmm_plan(nb.make_desc(M=256, N=128, K=128, ab_type="f16", cd_type="f16", ldb=128, ldd=256))
    with pytest.raises(nb.NmError) as e:
        nb.nm_spmm_search(plan, 1.0, FAKE, FAKE, FAKE, 0.0, None, FAKE, repeats=0, stream=0)
    assert e.value.status == nb.NM_ERR_INVALID_ARG
    with pytest.raises(nb.NmError) as e:  # beta != 0 with C aliasing D
        nb.nm_spmm_search(plan, 1.0, FAKE, FAKE, FAKE, 0.5, FAKE, FAKE, stream=0)
    assert e.value.status == nb.NM_ERR_INVALID_ARG
    plan.destroy()
    # a plan that fixed its algorithm, an odd number of row blocks, or a CUDA-core product: nothing is
    # run (no GPU needed) and the plan's own choice is reported
    fixed = nb.nm_spmm_plan(nb.make_desc(M=256, N=128, K=128, ab_type="f16", cd_type="f16", ldb=128, ldd=256,
                                         algo=nb.NM_ALGO_SINGLE))
    assert nb.nm_spmm_search(fixed, 1.0, FAKE, FAKE, FAKE, 0.0, None, FAKE, stream=0) == nb.NM_ALGO_SINGLE
    odd = nb.nm_spmm_plan(nb.make_desc(M=384, N=128, K=128, ab_type="f16", cd_type="f16", ldb=128, ldd=384))
    assert nb.nm_spmm_search(odd, 1.0, FAKE, FAKE, FAKE, 0.0, None, FAKE, stream=0) == nb.NM_ALGO_DEFAULT
    gather = nb.nm_spmm_plan(nb.make_desc(M=256, N=8, K=256, n=8, m=32, ab_type="f16", cd_type="f16", ldb=256,
                                          ldd=256, meta_layout=nb.NM_META_CANONICAL))
    assert nb.nm_spmm_search(gather, 1.0, FAKE, FAKE, FAKE, 0.0, None, FAKE, stream=0) == nb.NM_ALGO_DEFAULT
    for p in (fixed, odd, gather):
        p.destroy()


def test_sgd_prune_argument_checks(lib):
    L = nb.lib()

    def call(W=FAKE, dW=FAKE + 4096, dtype=nb.NM_BF16, rows=64, cols=64, ld=64, ld_grad=64):
        return L.nm_sgd_prune_transposable(W, dW, 0.1, rows, cols, ld, ld_grad, dtype, None, None, None, None, None,
                                           nb.NM_META_TC, None)

    assert call(dtype=nb.NM_I8) == nb.NM_ERR_UNSUPPORTED
    assert call(dW=FAKE) == nb.NM_ERR_INVALID_ARG          # the gradient may not alias the weight
    assert call(dW=FAKE + 4098) == nb.NM_ERR_MISALIGNED    # four-element alignment of dW
    assert call(ld_grad=66) == nb.NM_ERR_MISALIGNED
    assert call(rows=62) == nb.NM_ERR_INVALID_ARG
    assert call(dW=None) == nb.NM_ERR_INVALID_ARG


def test_sparse_layer_validates_before_touching_the_device():
    import torch

    from structured_sparse_gemm_nm_gb300.sparse_linear import SemiStructuredSparseLinear

    with pytest.raises(ValueError):
        SemiStructuredSparseLinear(100, 64)          # not a multiple of 32
    with pytest.raises(ValueError):
        SemiStructuredSparseLinear(64, 64, dtype=torch.float32)
    with pytest.raises(ValueError):
        SemiStructuredSparseLinear(64, 64, device="cpu")  # no CPU path


def test_plan_launches(lib):
    """Kernels one nm_spmm call launches: the masked dW sums two K splits inside the paired
    product (one launch), more splits or single CTAs add the finalize; other products launch one."""
    def dw_plan(o, i, T, algo=nb.NM_ALGO_DEFAULT):
        return nb.nm_spmm_plan(nb.make_desc(M=o, N=i, K=T, mode=nb.NM_SPMM_DENSE_MASKED, ab_type="bf16",
                                            cd_type="bf16", order_a=nb.NM_COL, order_b=nb.NM_ROW, order_cd=nb.NM_ROW,
                                            lda=o, ldb=i, ldd=i, meta_layout=nb.NM_META_CANONICAL, algo=algo))
    cases = [(dw_plan(3072, 768, 16384), 1, 2),                      # two splits, paired
             (dw_plan(3072, 768, 16384, nb.NM_ALGO_SINGLE), 2, 2),   # two splits, single CTAs: finalize
             (dw_plan(768, 768, 16384), 2, 7),                       # seven splits: finalize
             (dw_plan(512, 520, 192), 1, 1),                         # no K split
             (nb.nm_spmm_plan(nb.make_desc(M=3072, N=16384, K=768, ab_type="bf16", cd_type="bf16", ldb=768,
                                           ldd=3072)), 1, 1),
             (nb.nm_spmm_plan(nb.make_desc(M=0, N=16, K=32, ab_type="f16", cd_type="f16", ldb=32, ldd=8)), 0, 1)]
    for plan, want, split in cases:
        assert nb.nm_spmm_plan_launches(plan) == want
        assert nb.nm_spmm_plan_split_k(plan) == split
        plan.destroy()
    with pytest.raises(nb.NmError):
        nb._check(lib.nm_spmm_plan_split_k(None, None), "nm_spmm_plan_split_k")
    with pytest.raises(nb.NmError):
        nb._check(lib.nm_spmm_plan_launches(None, None), "nm_spmm_plan_launches")
