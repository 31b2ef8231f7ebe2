"""GPU check of nm_prune_vector_wise_noalloc, the vector-wise pruning entry
point that uses the library's fixed device scratch instead of a workspace
from the caller (for callers that may not allocate device memory when they
prune).  Its outputs must equal those of nm_prune_vector_wise, which takes a
caller workspace, on two calls in a row: the second call must not see
anything the first one left in the shared scratch.

This file is named so that pytest collects it last."""
import numpy as np
import pytest
import torch

from structured_sparse_gemm_nm_gb300 import binding as nb
from structured_sparse_gemm_nm_gb300 import inputs

from gpu_util import DEV, ensure_lib, u32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_lib()


ESIZE = {"f16": 2, "i8": 1}


def outputs(rows, cols, ld, keep, dtype):
    def buf(nbytes, fill):
        t = torch.empty(max(16, (nbytes + 15) // 16 * 16), dtype=torch.uint8, device=DEV)
        t.fill_(fill)
        return t

    es = ESIZE[dtype]
    return dict(W_out=buf(rows * ld * es, 0xAB), mask=buf(rows * (cols // 32) * 4, 0xCD),
                csr=buf((rows + 1 + keep) * 4, 0xEF), vals=buf(max(1, keep) * 32 * es, 0x5A))


def host(o, rows, cols, ld, keep, dtype):
    es = ESIZE[dtype]
    W_out = o["W_out"].cpu().numpy()[: rows * ld * es].reshape(rows, ld * es)[:, : cols * es]
    return dict(W_out=W_out, mask=u32(o["mask"], rows * (cols // 32)), csr=u32(o["csr"], rows + 1 + keep),
                vals=o["vals"].cpu().numpy()[: keep * 32 * es])


def with_workspace(W, rows, cols, ld, keep, score, dtype):
    o = outputs(rows, cols, ld, keep, dtype)
    wsb = nb.nm_prune_units_workspace(rows, cols, 1, 32)
    ws = torch.empty(max(16, wsb), dtype=torch.uint8, device=DEV)
    nb.nm_prune_vector_wise(W, rows, cols, ld, dtype, 32, keep, score, W_out=o["W_out"], ld_out=ld,
                            mask_bits=o["mask"], csr=o["csr"], vals=o["vals"], workspace=ws, workspace_bytes=wsb)
    torch.cuda.synchronize()
    return host(o, rows, cols, ld, keep, dtype)


def without_allocation(W, rows, cols, ld, keep, score, dtype):
    o = outputs(rows, cols, ld, keep, dtype)
    nb.nm_prune_vector_wise_noalloc(W, rows, cols, ld, dtype, 32, keep, score, W_out=o["W_out"], ld_out=ld,
                                    mask_bits=o["mask"], csr=o["csr"], vals=o["vals"])
    torch.cuda.synchronize()
    return host(o, rows, cols, ld, keep, dtype)


def make_weight(rows, cols, ld, dtype, seed):
    """rows x cols weight inside a rows x ld allocation (the padding holds values the call must not read)."""
    if dtype == "i8":
        full = inputs.uniform_int8((rows, ld), seed)
    else:
        full = inputs.normal((rows, ld), 0.02, seed, "f16")
    return full.to(DEV)


def test_noalloc_matches_workspace_entry_point_twice():
    # different problems back to back through the shared scratch, the largest first so that
    # each later one runs over what the earlier ones left behind: f16 and int8, a row pitch
    # wider than the row, and a call that keeps nothing
    cases = [  # rows, cols, ld, density, score, dtype, seed
        (4096, 4096, 4096, 0.25, nb.NM_SCORE_ABS_OF_SUM, "f16", 91),
        (300, 640, 640, 0.4, nb.NM_SCORE_SUM_OF_ABS, "f16", 92),
        (512, 1024, 1024, 0.3, nb.NM_SCORE_ABS_OF_SUM, "i8", 93),
        (200, 512, 576, 0.25, nb.NM_SCORE_SUM_OF_ABS, "f16", 94),
        (128, 256, 256, 0.0, nb.NM_SCORE_ABS_OF_SUM, "f16", 95),
    ]
    for rows, cols, ld, density, score, dtype, seed in cases:
        W = make_weight(rows, cols, ld, dtype, seed)
        keep = int(rows * cols // 32 * density)
        want = with_workspace(W, rows, cols, ld, keep, score, dtype)
        got = without_allocation(W, rows, cols, ld, keep, score, dtype)
        for k in ("mask", "csr", "vals", "W_out"):
            assert np.array_equal(got[k], want[k]), f"{rows}x{cols} {dtype}: {k} differs"
        if keep == 0:
            assert not got["mask"].any() and (got["csr"] == 0).all()


def test_noalloc_rejects_sizes_beyond_its_scratch():
    rows, cols = 4096, 4096 + 32  # one vector per row more than the fixed scratch holds
    assert rows * cols // 32 > nb.NM_NOALLOC_MAX_UNITS
    W = torch.empty((rows, cols), dtype=torch.float16, device=DEV)
    with pytest.raises(nb.NmError) as e:
        nb.nm_prune_vector_wise_noalloc(W, rows, cols, cols, "f16", 32, 1)
    assert e.value.status == nb.NM_ERR_UNSUPPORTED
