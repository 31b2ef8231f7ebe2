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


def outputs(rows, cols, keep):
    def buf(nbytes, fill):
        t = torch.empty(max(16, (nbytes + 15) // 16 * 16), dtype=torch.uint8, device=DEV)
        t.fill_(fill)
        return t

    return dict(W_out=buf(rows * cols * 2, 0xAB), mask=buf(rows * (cols // 32) * 4, 0xCD),
                csr=buf((rows + 1 + keep) * 4, 0xEF), vals=buf(max(1, keep) * 64, 0x5A))


def host(o, rows, cols, keep):
    return dict(W_out=o["W_out"].cpu().numpy()[: rows * cols * 2],
                mask=u32(o["mask"], rows * (cols // 32)),
                csr=u32(o["csr"], rows + 1 + keep),
                vals=o["vals"].cpu().numpy()[: keep * 64])


def with_workspace(W, rows, cols, keep, score):
    o = outputs(rows, cols, keep)
    wsb = nb.nm_prune_units_workspace(rows, cols, 1, 32)
    ws = torch.empty(wsb, dtype=torch.uint8, device=DEV)
    nb.nm_prune_vector_wise(W, rows, cols, cols, "f16", 32, keep, score, W_out=o["W_out"], ld_out=cols,
                            mask_bits=o["mask"], csr=o["csr"], vals=o["vals"], workspace=ws, workspace_bytes=wsb)
    torch.cuda.synchronize()
    return host(o, rows, cols, keep)


def without_allocation(W, rows, cols, keep, score):
    o = outputs(rows, cols, keep)
    nb.nm_prune_vector_wise_noalloc(W, rows, cols, cols, "f16", 32, keep, score, W_out=o["W_out"], ld_out=cols,
                                    mask_bits=o["mask"], csr=o["csr"], vals=o["vals"])
    torch.cuda.synchronize()
    return host(o, rows, cols, keep)


def test_noalloc_matches_workspace_entry_point_twice():
    # two different problems back to back through the shared scratch, the
    # larger first so that the second runs over what the first left behind
    cases = [(4096, 4096, 0.25, nb.NM_SCORE_ABS_OF_SUM, 91), (300, 640, 0.4, nb.NM_SCORE_SUM_OF_ABS, 92)]
    for rows, cols, density, score, seed in cases:
        W = inputs.normal((rows, cols), 0.02, seed, "f16").to(DEV)
        keep = int(rows * cols // 32 * density)
        want = with_workspace(W, rows, cols, keep, score)
        got = without_allocation(W, rows, cols, keep, score)
        for k in ("mask", "csr", "vals", "W_out"):
            assert np.array_equal(got[k], want[k]), f"{rows}x{cols}: {k} differs"


def test_noalloc_rejects_sizes_beyond_its_scratch():
    rows, cols = 4096, 4096 + 32  # one vector per row more than the fixed scratch holds
    assert rows * cols // 32 > nb.NM_NOALLOC_MAX_UNITS
    W = torch.empty((rows, cols), dtype=torch.float16, device=DEV)
    with pytest.raises(nb.NmError) as e:
        nb.nm_prune_vector_wise_noalloc(W, rows, cols, cols, "f16", 32, 1)
    assert e.value.status == nb.NM_ERR_UNSUPPORTED
