"""GPU parity of pruning, compression, decompression, check and the
transposable mask against the CPU oracle: bit-exact on every output byte."""
import numpy as np
import pytest
import torch

import oracle as o
from structured_sparse_gemm_nm_gb300 import binding as nb
from structured_sparse_gemm_nm_gb300 import inputs

from gpu_util import DEV, ESIZE, bits_of, dev_bytes, ensure_lib, to_dev_bits, u16, u32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_lib()


def host_matrix(rows, cols, dtype, seed, kind="normal"):
    """Seeded host matrix as bit patterns, with special values planted for kind='special'."""
    if dtype == "i8":
        return inputs.as_numpy_bits(inputs.uniform_int8((rows, cols), seed, -128, 127))
    if kind == "uniform":
        return inputs.as_numpy_bits(inputs.uniform((rows, cols), -1.0, 1.0, seed, dtype))
    if kind == "tiny":  # subnormal magnitudes (and a few normals) must order exactly
        rng = np.random.default_rng(seed)
        scale = 3e-5 if dtype == "f16" else 1e-38
        vals = (rng.standard_normal((rows, cols)) * scale).astype(np.float32)
        if dtype == "f16":
            return vals.astype(np.float16).view(np.uint16)
        return (vals.view(np.uint32) >> 16).astype(np.uint16)
    if kind == "ties":  # few distinct magnitudes: most tiles hold several best patterns
        rng = np.random.default_rng(seed)
        pool = np.array([0.0, 0.25, -0.25, 0.5, -0.5, 1.0, -1.0], dtype=np.float32)
        vals = rng.choice(pool, size=(rows, cols))
        if dtype == "f16":
            return vals.astype(np.float16).view(np.uint16)
        return (vals.view(np.uint32) >> 16).astype(np.uint16)
    a = inputs.as_numpy_bits(inputs.normal((rows, cols), 0.02, seed, dtype)).copy()
    if kind == "special":
        rng = np.random.default_rng(seed)
        pool = np.array([0.0, -0.0, 0.5, -0.5, 1.0, -1.0, np.inf, -np.inf, np.nan], dtype=np.float32)
        vals = rng.choice(pool, size=a.size // 3)
        if dtype == "f16":
            sb = vals.astype(np.float16).view(np.uint16)
        else:
            sb = (vals.view(np.uint32) >> 16).astype(np.uint16)
        idx = rng.choice(a.size, size=vals.size, replace=False)
        a.reshape(-1)[idx] = sb
    return a


def with_ld(a: np.ndarray, ld: int, dtype: str):
    """Device copy of `a` inside rows of `ld` elements; returns (tensor, padded host array)."""
    rows, cols = a.shape
    pad = np.zeros((rows, ld), dtype=a.dtype)
    pad[:, :cols] = a
    if ld > cols:
        pad[:, cols:] = 0x3C00 if dtype != "i8" else 7  # must stay untouched
    return to_dev_bits(pad, dtype), pad


# ------------------------------------------------------------------ nm_prune
PRUNE_CASES = [
    # rows, cols, ld, dtype, n, m, kind
    (64, 128, 128, "f16", 2, 4, "uniform"),
    (256, 512, 512, "f16", 2, 4, "normal"),
    (4096, 4096, 4096, "f16", 2, 4, "normal"),
    (300, 1024, 1032, "bf16", 2, 4, "special"),
    (37, 20, 20, "f16", 2, 4, "special"),
    (33, 52, 60, "bf16", 2, 4, "normal"),
    (128, 256, 256, "i8", 2, 4, "normal"),
    (19, 36, 40, "i8", 2, 4, "normal"),
    (4096, 4096, 4096, "f16", 8, 32, "normal"),
    (512, 4096, 4096, "f16", 4, 32, "normal"),
    (512, 4096, 4096, "f16", 16, 32, "normal"),
    (70, 96, 100, "bf16", 8, 32, "special"),     # generic path (ld not a multiple of 8)
    (70, 96, 104, "bf16", 8, 32, "special"),     # n:32 fast path with NaN/Inf groups
    (33, 128, 128, "f16", 16, 32, "special"),
    (40, 64, 64, "bf16", 4, 32, "normal"),
    (110000, 96, 96, "f16", 8, 32, "normal"),    # n:32 grid stride over rows of three groups
    (64, 256, 256, "f16", 4, 32, "tiny"),        # n:32 with subnormal keys
    (64, 256, 256, "bf16", 4, 32, "tiny"),
    (64, 256, 256, "f16", 8, 32, "tiny"),
    (64, 256, 256, "bf16", 8, 32, "tiny"),
    (64, 256, 256, "bf16", 16, 32, "tiny"),
    (128, 256, 256, "bf16", 4, 32, "ties"),      # n:32 with many equal keys at the threshold
    (128, 256, 256, "f16", 8, 32, "ties"),
    (45, 40, 40, "f16", 3, 8, "special"),
    (64, 64, 64, "i8", 1, 4, "normal"),
    (50, 30, 30, "f16", 2, 5, "normal"),
]


@pytest.mark.parametrize("rows,cols,ld,dtype,n,m,kind", PRUNE_CASES)
def test_prune_matches_oracle(rows, cols, ld, dtype, n, m, kind):
    a = host_matrix(rows, cols, dtype, seed=rows * 7 + cols + n, kind=kind)
    W, padded = with_ld(a, ld, dtype)
    out = W.clone()  # padding columns must come back untouched
    mask = dev_bytes(rows * ((cols + 31) // 32) * 4, fill=0xAB)
    nb.nm_prune(W, rows, cols, ld, dtype, n, m, out, ld, mask)
    torch.cuda.synchronize()
    want, want_mask = o.nm_prune(a, dtype, n, m)
    got = bits_of(out, dtype, (rows, ld))
    assert (got[:, :cols] == want).all()
    assert (got[:, cols:] == padded[:, cols:]).all()
    assert (u32(mask, rows * ((cols + 31) // 32)).reshape(rows, -1) == o.mask_to_bits(want_mask)).all()
    # in place
    nb.nm_prune(W, rows, cols, ld, dtype, n, m, W, ld, None)
    torch.cuda.synchronize()
    assert (bits_of(W, dtype, (rows, ld))[:, :cols] == want).all()


COMPRESS_CASES = [
    (64, 128, "f16", 2, 4, 0, nb.NM_META_CANONICAL),
    (64, 128, "f16", 2, 4, 0, nb.NM_META_TC),
    (300, 1024, "bf16", 2, 4, 0, nb.NM_META_TC),
    (4096, 4096, "f16", 2, 4, 0, nb.NM_META_TC),
    (4096, 4096, "bf16", 2, 4, 0, nb.NM_META_CANONICAL),
    (200, 96, "f16", 2, 4, 0, nb.NM_META_TC),
    (136, 4128, "bf16", 2, 4, 0, nb.NM_META_CANONICAL),  # word count not a multiple of the warp's
    (37, 20, "f16", 2, 4, 0, nb.NM_META_CANONICAL),
    (128, 256, "i8", 2, 4, 0, nb.NM_META_CANONICAL),
    (256, 512, "f16", 2, 4, 1, nb.NM_META_TC),
    (96, 44, "bf16", 2, 4, 1, nb.NM_META_CANONICAL),
    (4096, 4096, "f16", 8, 32, 0, nb.NM_META_CANONICAL),
    (4096, 4096, "f16", 4, 32, 0, nb.NM_META_CANONICAL),
    (4096, 4096, "f16", 16, 32, 0, nb.NM_META_CANONICAL),
    (64, 96, "bf16", 8, 32, 1, nb.NM_META_CANONICAL),
    (96, 256, "bf16", 16, 32, 0, nb.NM_META_CANONICAL),
    (50, 64, "f16", 4, 32, 0, nb.NM_META_CANONICAL),
    (45, 40, "f16", 3, 8, 0, nb.NM_META_CANONICAL),
]


@pytest.mark.parametrize("rows,cols,dtype,n,m,transpose,layout", COMPRESS_CASES)
def test_compress_decompress_match_oracle(rows, cols, dtype, n, m, transpose, layout):
    a = host_matrix(rows, cols, dtype, seed=rows + cols * 3 + n, kind="special" if dtype != "i8" else "normal")
    W = to_dev_bits(a, dtype)
    rl, cl = (cols, rows) if transpose else (rows, cols)
    vb, mb = nb.nm_compressed_size(rl, cl, dtype, n, m, layout)
    vals, meta = dev_bytes(vb, 0xCD), dev_bytes(mb, 0xCD)
    nb.nm_compress(W, rows, cols, cols, dtype, n, m, transpose, layout, vals, meta)
    torch.cuda.synchronize()
    ov, om = o.nm_compress(a, dtype, n, m, transpose=bool(transpose))
    assert (bits_of(vals, dtype, ov.shape) == ov).all()
    if (n, m) != (2, 4):
        assert (meta.cpu().numpy()[:mb] == om.reshape(-1)).all()
    elif layout == nb.NM_META_TC:
        want_tc = o.meta_to_tc_layout(om, rl, cl)
        assert (u32(meta, mb // 4).reshape(want_tc.shape) == want_tc).all()
    else:
        assert (u16(meta, mb // 2).reshape(rl, -1) == om).all()
    # decompress back to the pruned matrix
    out = torch.empty(rl * cl * ESIZE[dtype], dtype=torch.uint8, device=DEV)
    nb.nm_decompress(vals, meta, rl, cl, dtype, n, m, layout, out, cl)
    torch.cuda.synchronize()
    src = np.ascontiguousarray(a.T) if transpose else a
    pruned, _ = o.nm_prune(src, dtype, n, m)
    assert (bits_of(out, dtype, (rl, cl)) == pruned).all()


@pytest.mark.parametrize("dtype,n,m,transposable", [("f16", 2, 4, 0), ("bf16", 2, 4, 1), ("i8", 2, 4, 1),
                                                     ("f16", 8, 32, 0), ("f16", 3, 8, 0)])
def test_check_matches_oracle(dtype, n, m, transposable):
    rows, cols = 96, 128 if m != 3 else 120
    a = host_matrix(rows, cols, dtype, seed=5, kind="special" if dtype != "i8" else "normal")
    cnt = torch.zeros(1, dtype=torch.int32, device=DEV)
    for mat in (a, o.nm_prune(a, dtype, n, m)[0]):
        W = to_dev_bits(mat, dtype)
        nb.nm_check(W, rows, cols, cols, dtype, n, m, transposable, cnt)
        torch.cuda.synchronize()
        assert int(cnt.item()) == o.nm_check(mat, dtype, n, m, transposable=bool(transposable))
    if transposable:
        tp = o.nm_prune_transposable(a, dtype)[0]
        nb.nm_check(to_dev_bits(tp, dtype), rows, cols, cols, dtype, 2, 4, 1, cnt)
        torch.cuda.synchronize()
        assert int(cnt.item()) == 0


@pytest.mark.parametrize("rows,cols,ld,dtype,transposable", [(37, 48, 48, "f16", 0), (36, 40, 56, "bf16", 1),
                                                            (4096, 4096, 4096, "f16", 1)])
def test_check_strips_ragged_and_strided(rows, cols, ld, dtype, transposable):
    a = host_matrix(rows, cols, dtype, seed=rows + cols, kind="special")
    W, _ = with_ld(a, ld, dtype)
    cnt = torch.zeros(1, dtype=torch.int32, device=DEV)
    for mat in (a, o.nm_prune(a, dtype, 2, 4)[0]):
        Wm, _ = with_ld(mat, ld, dtype)
        nb.nm_check(Wm, rows, cols, ld, dtype, 2, 4, transposable, cnt)
        torch.cuda.synchronize()
        assert int(cnt.item()) == o.nm_check(mat, dtype, 2, 4, transposable=bool(transposable))


# ------------------------------------------------------------ transposable
TRANS_CASES = [
    (256, 512, "f16", nb.NM_META_TC, "normal"),       # SparseLinear 512 -> 256
    (2304, 768, "bf16", nb.NM_META_TC, "normal"),     # GPT-neo QKV
    (768, 768, "bf16", nb.NM_META_TC, "normal"),      # GPT-neo O
    (3072, 768, "bf16", nb.NM_META_TC, "normal"),     # GPT-neo FC1
    (768, 3072, "bf16", nb.NM_META_TC, "normal"),     # GPT-neo FC2
    (44, 20, "f16", nb.NM_META_CANONICAL, "special"),
    (96, 160, "bf16", nb.NM_META_TC, "special"),
    (64, 96, "i8", nb.NM_META_CANONICAL, "normal"),
    (512, 512, "f16", nb.NM_META_TC, "ties"),         # equal scores: the first pattern must win
    (68, 200, "bf16", nb.NM_META_CANONICAL, "ties"),
]


@pytest.mark.parametrize("rows,cols,dtype,layout,kind", TRANS_CASES)
def test_transposable_matches_oracle(rows, cols, dtype, layout, kind):
    a = host_matrix(rows, cols, dtype, seed=rows + 2 * cols, kind=kind)
    ld = cols + (8 if cols % 8 == 0 else 4)
    W, padded = with_ld(a, ld, dtype)
    out = W.clone()  # padding columns must come back untouched
    mask = dev_bytes(rows * ((cols + 31) // 32) * 4, 0xEE)
    vb, mb = nb.nm_compressed_size(rows, cols, dtype, 2, 4, layout)
    vbT, mbT = nb.nm_compressed_size(cols, rows, dtype, 2, 4, layout)
    vals, meta, valsT, metaT = dev_bytes(vb, 1), dev_bytes(mb, 1), dev_bytes(vbT, 1), dev_bytes(mbT, 1)
    nb.nm_prune_transposable(W, rows, cols, ld, dtype, out, ld, mask, vals, meta, valsT, metaT, layout)
    torch.cuda.synchronize()
    pruned, m_ref, (v, mt), (vT, mtT) = o.nm_prune_transposable(a, dtype)
    got = bits_of(out, dtype, (rows, ld))
    assert (got[:, :cols] == pruned).all()
    assert (got[:, cols:] == padded[:, cols:]).all()
    assert (u32(mask, rows * ((cols + 31) // 32)).reshape(rows, -1) == o.mask_to_bits(m_ref)).all()
    assert (bits_of(vals, dtype, v.shape) == v).all()
    assert (bits_of(valsT, dtype, vT.shape) == vT).all()
    if layout == nb.NM_META_TC:
        want_tc, want_tcT = o.meta_to_tc_layout(mt, rows, cols), o.meta_to_tc_layout(mtT, cols, rows)
        assert (u32(meta, mb // 4).reshape(want_tc.shape) == want_tc).all()
        assert (u32(metaT, mbT // 4).reshape(want_tcT.shape) == want_tcT).all()
    else:
        assert (u16(meta, mb // 2).reshape(rows, -1) == mt).all()
        assert (u16(metaT, mbT // 2).reshape(cols, -1) == mtT).all()


def test_empty_inputs_are_no_ops():
    W = dev_bytes(64)
    nb.nm_prune(W, 0, 32, 32, "f16", 2, 4, W, 32, None)
    nb.nm_compress(W, 0, 32, 32, "f16", 2, 4, 0, nb.NM_META_CANONICAL, None, None)
    nb.nm_prune_transposable(W, 0, 0, 1, "f16")
    cnt = torch.full((1,), 9, dtype=torch.int32, device=DEV)
    nb.nm_check(W, 0, 32, 32, "f16", 2, 4, 0, cnt)
    torch.cuda.synchronize()
    assert int(cnt.item()) == 0
