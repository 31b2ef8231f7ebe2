"""Python binding of the C ABI in ``include/nm.h`` (ctypes, argument marshalling only).

Function names match the C entry points.  Matrix arguments may be given as
torch tensors (their ``data_ptr()`` is passed), integer device addresses or
``None`` for a NULL pointer.  ``stream`` may be a ``torch.cuda.Stream``, a raw
``cudaStream_t`` integer or ``None`` for torch's current stream.  A non-OK
status raises :class:`NmError`.  Every step of the computation runs in the
CUDA library; nothing here computes.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "lib", "libnm.so")

# enums (include/nm.h)
NM_OK, NM_ERR_INVALID_ARG, NM_ERR_UNSUPPORTED, NM_ERR_MISALIGNED, NM_ERR_CUDA, NM_ERR_TIMEOUT = range(6)
NM_F16, NM_BF16, NM_I8, NM_F32, NM_I32 = range(5)
NM_META_CANONICAL, NM_META_TC = 0, 1
NM_SPMM_SPARSE_A, NM_SPMM_DENSE_MASKED, NM_SPMM_BLOCK_SPARSE_A = 0, 1, 2
NM_SCORE_ABS_OF_SUM, NM_SCORE_SUM_OF_ABS = 0, 1
NM_ROW, NM_COL = 0, 1

DTYPE_NAMES = {"f16": NM_F16, "bf16": NM_BF16, "i8": NM_I8, "f32": NM_F32, "i32": NM_I32}

NM_ALGO_DEFAULT, NM_ALGO_PAIRED, NM_ALGO_SINGLE = 0, 1, 2

# Every symbol include/nm.h declares.
EXPORTED = (
    "nm_status_string", "nm_version", "nm_last_cuda_error", "nm_compressed_size", "nm_prune", "nm_compress",
    "nm_prune_compress", "nm_decompress",
    "nm_check", "nm_prune_transposable", "nm_sgd_prune_transposable", "nm_prune_units_workspace", "nm_prune_vector_wise",
    "nm_prune_block_wise", "nm_prune_vector_wise_noalloc", "nm_spmm_plan", "nm_spmm_plan_workspace",
    "nm_spmm_plan_launches", "nm_spmm_plan_split_k", "nm_spmm_plan_destroy", "nm_spmm", "nm_spmm_search",
)
# Every symbol include/nm_testing.h declares.
TESTING_EXPORTED = ("nm_test_i8_sparse_mma_rate", "nm_test_spmm_wait_timeout")


class NmError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)}")


class SpmmDesc(ctypes.Structure):
    _fields_ = [
        ("M", ctypes.c_int64), ("N", ctypes.c_int64), ("K", ctypes.c_int64),
        ("mode", ctypes.c_int), ("n", ctypes.c_int), ("m", ctypes.c_int),
        ("ab_type", ctypes.c_int), ("cd_type", ctypes.c_int),
        ("order_a", ctypes.c_int), ("order_b", ctypes.c_int), ("order_cd", ctypes.c_int),
        ("lda", ctypes.c_int64), ("ldb", ctypes.c_int64), ("ldc", ctypes.c_int64), ("ldd", ctypes.c_int64),
        ("meta_layout", ctypes.c_int),
        ("algo", ctypes.c_int),
    ]


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded CUDA library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with `python -m structured_sparse_gemm_nm_gb300.build` "
                "(there is no fallback implementation)")
        L = ctypes.CDLL(LIB_PATH)
        i64, i32, vp, sz = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t
        L.nm_status_string.restype = ctypes.c_char_p
        L.nm_status_string.argtypes = [i32]
        L.nm_version.restype = i32
        L.nm_version.argtypes = []
        L.nm_last_cuda_error.restype = ctypes.c_char_p
        L.nm_last_cuda_error.argtypes = []
        sigs = {
            "nm_compressed_size": [i64, i64, i32, i32, i32, i32, ctypes.POINTER(sz), ctypes.POINTER(sz)],
            "nm_prune": [vp, i64, i64, i64, i32, i32, i32, vp, i64, vp, vp],
            "nm_compress": [vp, i64, i64, i64, i32, i32, i32, i32, i32, vp, vp, vp],
            "nm_prune_compress": [vp, i64, i64, i64, i32, i32, i32, vp, i64, vp, i32, vp, vp, vp],
            "nm_decompress": [vp, vp, i64, i64, i32, i32, i32, i32, vp, i64, vp],
            "nm_check": [vp, i64, i64, i64, i32, i32, i32, i32, vp, vp],
            "nm_prune_transposable": [vp, i64, i64, i64, i32, vp, i64, vp, vp, vp, vp, vp, i32, vp],
            "nm_sgd_prune_transposable": [vp, vp, ctypes.c_float, i64, i64, i64, i64, i32, vp, vp, vp, vp, vp, i32,
                                          vp],
            "nm_prune_units_workspace": [i64, i64, i32, i32, ctypes.POINTER(sz)],
            "nm_prune_vector_wise": [vp, i64, i64, i64, i32, i32, i64, i32, vp, i64, vp, vp, vp, vp, sz, vp],
            "nm_prune_block_wise": [vp, i64, i64, i64, i32, i32, i32, i64, vp, i64, vp, vp, vp, vp, sz, vp],
            "nm_prune_vector_wise_noalloc": [vp, i64, i64, i64, i32, i32, i64, i32, vp, i64, vp, vp, vp, vp],
            "nm_spmm_plan": [ctypes.POINTER(vp), ctypes.POINTER(SpmmDesc)],
            "nm_spmm_plan_workspace": [vp, ctypes.POINTER(sz)],
            "nm_spmm_plan_launches": [vp, ctypes.POINTER(i32)],
            "nm_spmm_plan_split_k": [vp, ctypes.POINTER(i32)],
            "nm_spmm_plan_destroy": [vp],
            "nm_spmm": [vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp, vp],
            "nm_spmm_search": [vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, i32, ctypes.POINTER(i32), vp],
            "nm_test_spmm_wait_timeout": [vp, ctypes.POINTER(SpmmDesc), vp, vp, vp, vp, vp, ctypes.c_longlong, vp],
            "nm_test_i8_sparse_mma_rate": [ctypes.c_int, ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_double)],
        }
        for name, args in sigs.items():
            f = getattr(L, name)
            f.restype = i32
            f.argtypes = args
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().nm_status_string(int(status)).decode()


def _ptr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x or None
    return x.data_ptr() or None


def _current_stream() -> int | None:
    """The current CUDA stream of the current device as a raw handle (NULL = legacy default)."""
    import torch

    raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
    if raw is not None:  # a third of the cost of building a torch.cuda.Stream object
        return raw(torch.cuda.current_device()) or None
    return torch.cuda.current_stream().cuda_stream or None


def _stream(s) -> int | None:
    if s is None:
        return _current_stream()
    if isinstance(s, int):
        return s or None
    return s.cuda_stream or None


def _dt(d) -> int:
    return DTYPE_NAMES[d] if isinstance(d, str) else int(d)


def _check(st: int, where: str) -> None:
    if st != NM_OK:
        if st == NM_ERR_CUDA:
            where = f"{where} ({lib().nm_last_cuda_error().decode()})"
        raise NmError(st, where)


# ------------------------------------------------------------------ calls
def nm_version() -> int:
    return lib().nm_version()


def nm_compressed_size(rows, cols, dtype, n, m, layout=NM_META_CANONICAL):
    vb, mb = ctypes.c_size_t(), ctypes.c_size_t()
    _check(lib().nm_compressed_size(rows, cols, _dt(dtype), n, m, layout, ctypes.byref(vb), ctypes.byref(mb)),
           "nm_compressed_size")
    return vb.value, mb.value


def nm_prune(W, rows, cols, ld, dtype, n, m, W_out=None, ld_out=0, mask_bits=None, stream=None):
    _check(lib().nm_prune(_ptr(W), rows, cols, ld, _dt(dtype), n, m, _ptr(W_out), ld_out, _ptr(mask_bits),
                          _stream(stream)), "nm_prune")


def nm_compress(W, rows, cols, ld, dtype, n, m, transpose=0, layout=NM_META_CANONICAL, vals=None, meta=None,
                stream=None):
    _check(lib().nm_compress(_ptr(W), rows, cols, ld, _dt(dtype), n, m, int(transpose), layout, _ptr(vals),
                             _ptr(meta), _stream(stream)), "nm_compress")


def nm_prune_compress(W, rows, cols, ld, dtype, n, m, W_out=None, ld_out=0, mask_bits=None,
                      layout=NM_META_CANONICAL, vals=None, meta=None, stream=None):
    _check(lib().nm_prune_compress(_ptr(W), rows, cols, ld, _dt(dtype), n, m, _ptr(W_out), ld_out, _ptr(mask_bits),
                                   layout, _ptr(vals), _ptr(meta), _stream(stream)), "nm_prune_compress")


def nm_decompress(vals, meta, rows, cols, dtype, n, m, layout, W_out, ld_out, stream=None):
    _check(lib().nm_decompress(_ptr(vals), _ptr(meta), rows, cols, _dt(dtype), n, m, layout, _ptr(W_out), ld_out,
                               _stream(stream)), "nm_decompress")


def nm_check(W, rows, cols, ld, dtype, n, m, transposable, d_violations, stream=None):
    _check(lib().nm_check(_ptr(W), rows, cols, ld, _dt(dtype), n, m, int(transposable), _ptr(d_violations),
                          _stream(stream)), "nm_check")


def nm_prune_transposable(W, rows, cols, ld, dtype, W_out=None, ld_out=0, mask_bits=None, vals=None, meta=None,
                          valsT=None, metaT=None, layout=NM_META_CANONICAL, stream=None):
    _check(lib().nm_prune_transposable(_ptr(W), rows, cols, ld, _dt(dtype), _ptr(W_out), ld_out, _ptr(mask_bits),
                                       _ptr(vals), _ptr(meta), _ptr(valsT), _ptr(metaT), layout, _stream(stream)),
           "nm_prune_transposable")


def nm_sgd_prune_transposable(W, dW, lr, rows, cols, ld, ld_grad, dtype, mask_bits=None, vals=None, meta=None,
                              valsT=None, metaT=None, layout=NM_META_CANONICAL, stream=None):
    """W <- W - lr * dW (in place), then W's transposable 2:4 mask and compressed forms, in one pass."""
    _check(lib().nm_sgd_prune_transposable(_ptr(W), _ptr(dW), float(lr), rows, cols, ld, ld_grad, _dt(dtype),
                                           _ptr(mask_bits), _ptr(vals), _ptr(meta), _ptr(valsT), _ptr(metaT), layout,
                                           _stream(stream)), "nm_sgd_prune_transposable")


def nm_prune_units_workspace(rows, cols, bh, bw) -> int:
    b = ctypes.c_size_t()
    _check(lib().nm_prune_units_workspace(rows, cols, bh, bw, ctypes.byref(b)), "nm_prune_units_workspace")
    return b.value


def nm_prune_vector_wise(W, rows, cols, ld, dtype, v, keep, score=NM_SCORE_ABS_OF_SUM, W_out=None, ld_out=0,
                         mask_bits=None, csr=None, vals=None, workspace=None, workspace_bytes=0, stream=None):
    _check(lib().nm_prune_vector_wise(_ptr(W), rows, cols, ld, _dt(dtype), v, int(keep), int(score), _ptr(W_out),
                                      ld_out, _ptr(mask_bits), _ptr(csr), _ptr(vals), _ptr(workspace),
                                      workspace_bytes, _stream(stream)), "nm_prune_vector_wise")


def nm_prune_block_wise(W, rows, cols, ld, dtype, bh, bw, keep, W_out=None, ld_out=0, mask_bits=None, csr=None,
                        vals=None, workspace=None, workspace_bytes=0, stream=None):
    _check(lib().nm_prune_block_wise(_ptr(W), rows, cols, ld, _dt(dtype), bh, bw, int(keep), _ptr(W_out), ld_out,
                                     _ptr(mask_bits), _ptr(csr), _ptr(vals), _ptr(workspace), workspace_bytes,
                                     _stream(stream)), "nm_prune_block_wise")


NM_NOALLOC_MAX_UNITS = 524288


def nm_prune_vector_wise_noalloc(W, rows, cols, ld, dtype, v, keep, score=NM_SCORE_ABS_OF_SUM, W_out=None, ld_out=0,
                                 mask_bits=None, csr=None, vals=None, stream=None):
    """nm_prune_vector_wise with the library's fixed scratch instead of a caller workspace."""
    _check(lib().nm_prune_vector_wise_noalloc(_ptr(W), rows, cols, ld, _dt(dtype), v, int(keep), int(score),
                                              _ptr(W_out), ld_out, _ptr(mask_bits), _ptr(csr), _ptr(vals),
                                              _stream(stream)), "nm_prune_vector_wise_noalloc")


class SpmmPlan:
    """Owns an ``nm_spmm_plan_t``; destroyed with the object or by :func:`nm_spmm_plan_destroy`."""

    def __init__(self, handle: int, desc: SpmmDesc):
        self.handle = handle
        self.desc = desc

    def destroy(self) -> None:
        if self.handle:
            lib().nm_spmm_plan_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.destroy()
        except Exception:
            pass


def make_desc(**kw) -> SpmmDesc:
    d = SpmmDesc()
    d.mode = NM_SPMM_SPARSE_A
    d.n, d.m = 2, 4
    d.order_a, d.order_b, d.order_cd = NM_ROW, NM_COL, NM_COL
    d.meta_layout = NM_META_TC
    for k, v in kw.items():
        if k in ("ab_type", "cd_type"):
            v = _dt(v)
        setattr(d, k, v)
    return d


def nm_spmm_plan(desc: SpmmDesc) -> SpmmPlan:
    h = ctypes.c_void_p()
    _check(lib().nm_spmm_plan(ctypes.byref(h), ctypes.byref(desc)), "nm_spmm_plan")
    return SpmmPlan(h.value, desc)


def nm_spmm_plan_workspace(plan: SpmmPlan) -> int:
    b = ctypes.c_size_t()
    _check(lib().nm_spmm_plan_workspace(plan.handle, ctypes.byref(b)), "nm_spmm_plan_workspace")
    return b.value


def nm_spmm_plan_launches(plan: SpmmPlan) -> int:
    n = ctypes.c_int32()
    _check(lib().nm_spmm_plan_launches(plan.handle, ctypes.byref(n)), "nm_spmm_plan_launches")
    return n.value


def nm_spmm_plan_split_k(plan: SpmmPlan) -> int:
    """K splits of a DENSE_MASKED plan (1 = not split; 1 for other products)."""
    n = ctypes.c_int32()
    _check(lib().nm_spmm_plan_split_k(plan.handle, ctypes.byref(n)), "nm_spmm_plan_split_k")
    return n.value


def nm_spmm_plan_destroy(plan: SpmmPlan) -> None:
    plan.destroy()


def _scalar(x, is_int: bool):
    return ctypes.c_int32(int(x)) if is_int else ctypes.c_float(float(x))


def nm_spmm(plan: SpmmPlan, alpha, A, A_meta, B, beta, C, D, workspace=None, workspace_bytes=0, d_status=None,
            stream=None):
    is_int = plan.desc.ab_type == NM_I8 and plan.desc.cd_type == NM_I32
    a, b = _scalar(alpha, is_int), _scalar(beta, is_int)
    _check(lib().nm_spmm(plan.handle, ctypes.byref(a), _ptr(A), _ptr(A_meta), _ptr(B), ctypes.byref(b), _ptr(C),
                         _ptr(D), _ptr(workspace), workspace_bytes, _ptr(d_status), _stream(stream)), "nm_spmm")


def nm_spmm_search(plan: SpmmPlan, alpha, A, A_meta, B, beta, C, D, workspace=None, workspace_bytes=0, repeats=3,
                   stream=None) -> int:
    """Times the candidate algorithms on these operands, keeps the fastest in the plan, returns it."""
    is_int = plan.desc.ab_type == NM_I8 and plan.desc.cd_type == NM_I32
    a, b = _scalar(alpha, is_int), _scalar(beta, is_int)
    chosen = ctypes.c_int()
    _check(lib().nm_spmm_search(plan.handle, ctypes.byref(a), _ptr(A), _ptr(A_meta), _ptr(B), ctypes.byref(b),
                                _ptr(C), _ptr(D), _ptr(workspace), workspace_bytes, int(repeats),
                                ctypes.byref(chosen), _stream(stream)), "nm_spmm_search")
    return chosen.value


def nm_test_spmm_wait_timeout(desc: SpmmDesc, A, A_meta, B, D, d_status, budget_cycles: int, stream=None):
    """Test hook: runs the sparse tensor-core kernel with one wait that can never complete."""
    _check(lib().nm_test_spmm_wait_timeout(None, ctypes.byref(desc), _ptr(A), _ptr(A_meta), _ptr(B), _ptr(D),
                                           _ptr(d_status), int(budget_cycles), _stream(stream)),
           "nm_test_spmm_wait_timeout")


def nm_test_i8_sparse_mma_rate(iters: int = 20000) -> float:
    """Measurement hook: the warp-level 2:4 sparse int8 MMA's rate on all SMs, in dense-equivalent TOPS."""
    ms, ops = ctypes.c_float(), ctypes.c_double()
    _check(lib().nm_test_i8_sparse_mma_rate(int(iters), ctypes.byref(ms), ctypes.byref(ops)),
           "nm_test_i8_sparse_mma_rate")
    return ops.value / ms.value / 1e9
