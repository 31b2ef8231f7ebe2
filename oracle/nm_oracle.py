"""CPU oracle for the N:M structured-sparsity hot path.

TEST INFRASTRUCTURE ONLY.  This module is imported by ``tests/``, by
``__graft_entry__.smoke()`` and by ``bench.py``'s CPU-baseline leg and
reference arm, never by the product (the CUDA library in
``structured_sparse_gemm_nm_gb300/`` and its Python binding).  It shares no
code, table or helper with that library.

It is deliberately plain: numpy, float64 for every floating-point result,
int64 for integer results, library primitives (``lexsort``, ``matmul``) used
only as whole steps.  Each function names the passage it follows.

Storage conventions (the same bytes the CUDA path reads and writes):

* ``f16`` and ``bf16`` matrices are numpy ``uint16`` arrays of bit patterns,
  ``i8`` matrices are numpy ``int8`` arrays.
* Groups of ``m`` are ``m`` consecutive elements of a row.
* 2:4 metadata ("canonical"): one 4-bit code per group, ``i0 | i1 << 2`` with
  ``i0 < i1`` the kept positions; group ``g`` of a row sits at bits
  ``4*(g % 4)`` of uint16 word ``g // 4``; ``ceil(cols / 16)`` words per row.
* Other N:M: one uint8 position per kept value, in the order of the values.
* Kept values are stored in ascending position order with their original
  bits; pruned slots of a dense output are +0.
* Bit masks: row-major, ``ceil(cols / 32)`` uint32 words per row, bit
  ``c % 32`` of word ``c // 32`` is element ``c``.

Readings where the pages are silent:

* ties in magnitude go to the lower position (``topk``'s tie order is
  unspecified);
* NaN ranks above every number, including +Inf (``topk`` treats NaN as the
  largest value); several NaNs tie;
* ``cols % m == 0`` is required (the page's ``reshape_1d`` is not shown);
* the transposable 4x4 mask is the one among the 90 patterns with two kept
  entries in every row and every column of the tile that has the largest
  float32 score ``((p0 + p1) + p2) + p3``, ``p_r`` being the float32 sum of
  the two kept magnitudes of row ``r``; ties go to the earliest pattern in
  the canonical order (row 0's pair outermost); NaN magnitudes score +Inf;
* an int8 GEMM produces an int32 ``D``; ``alpha`` and ``beta`` are int32 and
  the arithmetic wraps modulo 2**32;
* ``beta == 0`` means ``C`` is not read.

Parity pins for each function live in ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import numpy as np

DTYPES = ("f16", "bf16", "i8")

# The six ways to keep 2 of 4 positions, in lexicographic order.  Used for
# the transposable 4x4 pattern enumeration.
PAIRS = ((0, 1), (0, 2), (0, 3), (1, 2), (1, 3), (2, 3))


# --------------------------------------------------------------------------
# element decoding
# --------------------------------------------------------------------------
def decode(x, dtype: str) -> np.ndarray:
    """Exact float64 values of stored elements (f16/bf16 bit patterns or int8)."""
    x = np.asarray(x)
    if dtype == "f16":
        return x.astype(np.uint16).view(np.float16).astype(np.float64)
    if dtype == "bf16":
        return (x.astype(np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    if dtype == "i8":
        return x.astype(np.int8).astype(np.float64)
    raise ValueError(dtype)


def _zero_like(W: np.ndarray) -> np.ndarray:
    return np.zeros_like(W)  # bit pattern 0 is +0 for f16/bf16 and 0 for int8


def _check_groups(cols: int, n: int, m: int) -> None:
    if not (1 <= n < m <= 32):
        raise ValueError(f"need 1 <= n < m <= 32, got n={n} m={m}")
    if cols % m:
        raise ValueError(f"cols={cols} is not a multiple of m={m}")


# --------------------------------------------------------------------------
# N:M greedy magnitude pruning
#   NVIDIA/apex PR #1631 "[sparse] update support for arbitrary N:M settings
#   sparse", extension 1 (``mn_1d_greedy``): per group of m consecutive
#   weights take ``abs().topk(n)`` and set those mask entries to 1.
#   cuSPARSELt blog, Figure 1 text: 2:4 means at least two of every four
#   elements are zero.
# --------------------------------------------------------------------------
def nm_mask(W: np.ndarray, dtype: str, n: int, m: int) -> np.ndarray:
    """Boolean mask keeping the n largest |w| of every m-group; ties to the lower position."""
    rows, cols = W.shape
    _check_groups(cols, n, m)
    v = decode(W, dtype).reshape(-1, m)
    nan = np.isnan(v)
    mag = np.where(nan, 0.0, np.abs(v))
    pos = np.broadcast_to(np.arange(m), v.shape)
    # lexsort: last key is primary.  Order: NaN first, then larger |w|, then lower position.
    order = np.lexsort((pos, -mag, -nan.astype(np.int8)), axis=-1)
    mask = np.zeros(v.shape, dtype=bool)
    np.put_along_axis(mask, order[:, :n], True, axis=1)
    return mask.reshape(rows, cols)


def nm_prune(W: np.ndarray, dtype: str, n: int, m: int):
    """Pruned copy of W (dropped slots +0) and its mask."""
    mask = nm_mask(W, dtype, n, m)
    return np.where(mask, W, _zero_like(W)), mask


def mask_to_bits(mask: np.ndarray) -> np.ndarray:
    """Row-major packed bit mask, ceil(cols/32) uint32 words per row."""
    rows, cols = mask.shape
    words = (cols + 31) // 32
    padded = np.zeros((rows, words * 32), dtype=np.uint64)
    padded[:, :cols] = mask
    weights = (np.uint64(1) << np.arange(32, dtype=np.uint64))
    return (padded.reshape(rows, words, 32) * weights).sum(axis=-1).astype(np.uint32)


def bits_to_mask(bits: np.ndarray, cols: int) -> np.ndarray:
    rows = bits.shape[0]
    b = bits.astype(np.uint64)[:, :, None] >> np.arange(32, dtype=np.uint64)
    return (b & np.uint64(1)).astype(bool).reshape(rows, -1)[:, :cols]


# --------------------------------------------------------------------------
# compression into values + metadata
#   cuSPARSELt blog, Figure 2 text: the pruned matrix is stored at half size
#   plus a small metadata array recording where the nonzeros were; the
#   metadata selects the matching entries of the other operand.
# --------------------------------------------------------------------------
def meta_words_per_row(cols: int) -> int:
    return (cols // 4 + 3) // 4


def compress_by_mask(W: np.ndarray, mask: np.ndarray, n: int, m: int):
    """Values (kept entries in ascending position) and metadata for a mask with exactly n kept per m-group."""
    rows, cols = W.shape
    _check_groups(cols, n, m)
    G = W.reshape(rows, cols // m, m)
    K = mask.reshape(rows, cols // m, m)
    if not (K.sum(axis=-1) == n).all():
        raise ValueError("mask does not keep exactly n entries in every group")
    # stable argsort of ~mask puts kept positions first, in ascending order
    pos = np.argsort(~K, axis=-1, kind="stable")[..., :n]
    vals = np.take_along_axis(G, pos, axis=-1).reshape(rows, (cols // m) * n)
    if (n, m) == (2, 4):
        code = (pos[..., 0] | (pos[..., 1] << 2)).astype(np.uint32)  # rows x groups
        groups = cols // 4
        words = meta_words_per_row(cols)
        padded = np.zeros((rows, words * 4), dtype=np.uint32)
        padded[:, :groups] = code
        shifts = np.array([0, 4, 8, 12], dtype=np.uint32)
        meta = (padded.reshape(rows, words, 4) << shifts).sum(axis=-1).astype(np.uint16)
    else:
        meta = pos.reshape(rows, (cols // m) * n).astype(np.uint8)
    return vals, meta


def nm_compress(W: np.ndarray, dtype: str, n: int, m: int, transpose: bool = False):
    """Compress W (or W^T) with the greedy selection applied to that matrix itself."""
    if transpose:
        W = np.ascontiguousarray(W.T)
    return compress_by_mask(W, nm_mask(W, dtype, n, m), n, m)


def meta_positions(meta: np.ndarray, rows: int, cols: int, n: int, m: int) -> np.ndarray:
    """Kept positions per group, shape rows x cols/m x n."""
    if (n, m) == (2, 4):
        groups = cols // 4
        w = meta.astype(np.uint32)
        codes = ((w[:, :, None] >> np.array([0, 4, 8, 12], dtype=np.uint32)) & 0xF).reshape(rows, -1)[:, :groups]
        return np.stack([codes & 3, (codes >> 2) & 3], axis=-1).astype(np.int64)
    return meta.reshape(rows, cols // m, n).astype(np.int64)


def nm_decompress(vals: np.ndarray, meta: np.ndarray, rows: int, cols: int, n: int, m: int) -> np.ndarray:
    """Scatter kept values back to their positions; every other slot is +0."""
    _check_groups(cols, n, m)
    out = np.zeros((rows, cols // m, m), dtype=vals.dtype)
    pos = meta_positions(meta, rows, cols, n, m)
    np.put_along_axis(out, pos, vals.reshape(rows, cols // m, n), axis=-1)
    return out.reshape(rows, cols)


# --------------------------------------------------------------------------
# pattern check
#   cuSPARSELt blog, code example (``cusparseLtSpMMAPruneCheck``): a nonzero
#   ``is_valid`` means the matrix does not conform to the sparsity pattern.
# --------------------------------------------------------------------------
def nm_check(W: np.ndarray, dtype: str, n: int, m: int, transposable: bool = False) -> int:
    """Number of m-groups holding more than n nonzeros (NaN counts as nonzero).

    With ``transposable`` the groups of 4 consecutive rows in every column
    (aligned to multiples of 4) are counted too."""
    rows, cols = W.shape
    _check_groups(cols, n, m)
    nz = decode(W, dtype) != 0
    bad = int((nz.reshape(-1, m).sum(axis=1) > n).sum())
    if transposable:
        if (n, m) != (2, 4) or rows % 4:
            raise ValueError("transposable check needs 2:4 and rows % 4 == 0")
        bad += int((nz.T.reshape(-1, 4).sum(axis=1) > 2).sum())
    return bad


# --------------------------------------------------------------------------
# transposable 4x4-tile 2:4 mask
#   PyTorch issue #126420, maintainer reply: sparsity is applied per 4x4
#   tile so that both W x (forward) and W^T dL/dy (backward) run on 2:4
#   sparse hardware, i.e. the mask is 2:4 along rows and along columns.
# --------------------------------------------------------------------------
def transposable_patterns():
    """The 4x4 0/1 patterns with two ones in every row and every column.

    Canonical order: row 0's pair is the outermost loop, rows' pairs run in
    lexicographic order.  Returns a list of (pair indices per row, 4x4 bool)."""
    pats = []
    for a in range(6):
        for b in range(6):
            for c in range(6):
                for d in range(6):
                    t = np.zeros((4, 4), dtype=bool)
                    for r, p in enumerate((a, b, c, d)):
                        t[r, list(PAIRS[p])] = True
                    if (t.sum(axis=0) == 2).all():
                        pats.append(((a, b, c, d), t))
    return pats


def transposable_mask(W: np.ndarray, dtype: str) -> np.ndarray:
    """Per 4x4 tile, the valid pattern with the largest float32 kept-magnitude score."""
    rows, cols = W.shape
    if rows % 4 or cols % 4:
        raise ValueError("rows and cols must be multiples of 4")
    v = decode(W, dtype)
    mag = np.where(np.isnan(v), np.inf, np.abs(v)).astype(np.float32)  # exact for f16/bf16/i8
    tiles = mag.reshape(rows // 4, 4, cols // 4, 4).transpose(0, 2, 1, 3).reshape(-1, 4, 4)
    # p[t, r, q]: float32 sum of the two magnitudes of pair q in row r
    p = np.stack([tiles[:, :, i] + tiles[:, :, j] for (i, j) in PAIRS], axis=-1).astype(np.float32)
    pats = transposable_patterns()
    scores = np.empty((tiles.shape[0], len(pats)), dtype=np.float32)
    for k, ((a, b, c, d), _) in enumerate(pats):
        s = p[:, 0, a] + p[:, 1, b]
        s = s + p[:, 2, c]
        s = s + p[:, 3, d]
        scores[:, k] = s
    best = np.argmax(scores, axis=1)  # first maximum = earliest pattern
    pat_masks = np.stack([t for (_, t) in pats])
    mt = pat_masks[best]  # tiles x 4 x 4
    return mt.reshape(rows // 4, cols // 4, 4, 4).transpose(0, 2, 1, 3).reshape(rows, cols)


def nm_prune_transposable(W: np.ndarray, dtype: str):
    """Pruned W, its mask, and the compressed forms of W (groups along rows) and W^T."""
    mask = transposable_mask(W, dtype)
    pruned = np.where(mask, W, _zero_like(W))
    vals, meta = compress_by_mask(W, mask, 2, 4)
    valsT, metaT = compress_by_mask(np.ascontiguousarray(W.T), np.ascontiguousarray(mask.T), 2, 4)
    return pruned, mask, (vals, meta), (valsT, metaT)


# --------------------------------------------------------------------------
# one training step's weight write with the run-time re-prune
#   PyTorch issue #126420, maintainer reply: fast sparsification kernels do
#   run-time sparsity for training; the layer keeps a dense master weight,
#   updates it, and derives the 4x4-tile 2:4 mask and the compressed forms of
#   W and W^T from the updated weight.
#   Reading (the pages give no optimizer): plain SGD, w <- w - lr * g, with
#   the product and the sum each rounded to float32 and the result rounded to
#   the weight's type (round to nearest even); finite inputs.
# --------------------------------------------------------------------------
def encode(x: np.ndarray, dtype: str) -> np.ndarray:
    """float32 values -> f16 / bf16 bit patterns, rounded to nearest even (finite values)."""
    x = np.asarray(x, dtype=np.float32)
    if dtype == "f16":
        return x.astype(np.float16).view(np.uint16)
    if dtype == "bf16":
        b = x.view(np.uint32).astype(np.uint64)
        rounded = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
        return rounded.astype(np.uint16)
    raise ValueError(dtype)


def sgd_update(W: np.ndarray, dW: np.ndarray, lr: float, dtype: str) -> np.ndarray:
    """w + (-lr * g): each operation rounded to float32, the result rounded to the element type."""
    if dtype not in ("f16", "bf16"):
        raise ValueError("the update is defined for f16 and bf16 weights")
    w = decode(W, dtype).astype(np.float32)  # exact
    g = decode(dW, dtype).astype(np.float32)  # exact
    nlr = -np.float32(lr)
    t = (nlr * g).astype(np.float32)
    return encode((w + t).astype(np.float32), dtype)


def sgd_prune_transposable(W: np.ndarray, dW: np.ndarray, lr: float, dtype: str):
    """The updated dense weight, then its transposable prune: (W_new, pruned, mask, (vals, meta), (valsT, metaT))."""
    W_new = sgd_update(W, dW, lr, dtype)
    return (W_new,) + tuple(nm_prune_transposable(W_new, dtype))


# --------------------------------------------------------------------------
# the sparse-dense product
#   cuSPARSELt blog, GEMM paragraph: D = alpha*op(A)*op(B) + beta*C with A
#   (M x K) the structured sparse operand, B (K x N), C = D (M x N); FP16 and
#   BF16 inputs accumulate in FP32, INT8 inputs in INT32 ("key features").
#   Sparse tensor cores skip the zeros, so the product equals the dense
#   product of the pruned matrix.
# --------------------------------------------------------------------------
def spmm(alpha: float, A: np.ndarray, B: np.ndarray, beta: float = 0.0, C=None) -> np.ndarray:
    """float64 D = alpha * A @ B + beta * C for float64 A (M x K, already pruned) and B (K x N)."""
    D = float(alpha) * (np.asarray(A, np.float64) @ np.asarray(B, np.float64))
    if beta != 0.0:
        D = D + float(beta) * np.asarray(C, np.float64)
    return D


def _wrap32(x: np.ndarray) -> np.ndarray:
    return ((x.astype(np.int64) + (1 << 31)) % (1 << 32) - (1 << 31)).astype(np.int32)


def spmm_int(alpha: int, A: np.ndarray, B: np.ndarray, beta: int = 0, C=None) -> np.ndarray:
    """int32 D = alpha * A @ B + beta * C for int8 A (M x K, pruned) and B (K x N), modulo 2**32."""
    acc = np.asarray(A, np.int64) @ np.asarray(B, np.int64)
    D = int(alpha) * acc
    if beta != 0:
        D = D + int(beta) * np.asarray(C, np.int64)
    return _wrap32(D)


def spmm_int8_out(alpha: float, A: np.ndarray, B: np.ndarray, beta: float = 0.0, C=None) -> np.ndarray:
    """int8 D from int8 A (M x K) and B (K x N) with float scales (cuSPARSELt blog, key features: INT8
    inputs and output; the scale and rounding are this library's reading, the pages give none):
    acc exact (int64; it must fit int32), converted to float32 (nearest even), alpha * acc and
    beta * C each rounded to float32, their sum rounded to float32, then to the nearest integer
    (ties to even) and clamped to [-128, 127]."""
    acc = A.astype(np.int64) @ B.astype(np.int64)
    if np.abs(acc).max(initial=0) >= 2 ** 31:
        raise ValueError("the int32 accumulator would overflow")
    x = (np.float32(alpha) * acc.astype(np.float32)).astype(np.float32)
    if C is not None:
        x = (x + (np.float32(beta) * C.astype(np.float32)).astype(np.float32)).astype(np.float32)
    return np.clip(np.rint(x), -128, 127).astype(np.int8)


def spmm_compressed(alpha: float, vals, meta, dtype: str, M: int, K: int, n: int, m: int, B, beta=0.0, C=None):
    """The product from the compressed form: decompress, then the dense definition."""
    A = decode(nm_decompress(vals, meta, M, K, n, m), dtype)
    return spmm(alpha, A, B, beta, C)


def masked_weight_grad(dY: np.ndarray, X: np.ndarray, mask: np.ndarray) -> np.ndarray:
    """dW = mask * (dY^T X) in float64 for dY (tokens x out), X (tokens x in), mask (out x in).

    The gradient of Y = X W^T with respect to W, restricted to the kept
    entries so that the updated weight keeps its sparsity pattern."""
    return np.where(mask, np.asarray(dY, np.float64).T @ np.asarray(X, np.float64), 0.0)


# --------------------------------------------------------------------------
# vector-wise and block-wise masks
#   NVIDIA/apex PR #1631, extension 2 (``unstructured_vector_wise``,
#   ``unstructured_block_wise``).
# --------------------------------------------------------------------------
def vector_wise_mask(W: np.ndarray, dtype: str, density: float, v: int = 32, score: str = "abs_of_sum") -> np.ndarray:
    """Keep the floor(#vectors * density) 1 x v vectors with the largest score.

    Vectors are consecutive v-element chunks of the row-major matrix.  The
    page scores a vector by the absolute value of its (signed) sum; the
    alternative ``sum_of_abs`` is offered for comparison.  Ties go to the
    lower vector index.  Sums are exact in float64 for f16 and int8 inputs.
    Special values follow float64 arithmetic: an infinite score ranks above
    every number, a NaN score (a NaN element, or +Inf and -Inf summed) below
    every number, including 0."""
    if dtype == "bf16":
        raise ValueError("vector-wise scores are exact only for f16 and int8")
    flat = decode(W, dtype).reshape(-1, v)
    nvec = flat.shape[0]
    keep = int(nvec * density)
    s = np.abs(flat.sum(axis=1)) if score == "abs_of_sum" else np.abs(flat).sum(axis=1)
    order = np.lexsort((np.arange(nvec), -s))
    kept = np.zeros(nvec, dtype=bool)
    kept[order[:keep]] = True
    return np.repeat(kept, v).reshape(W.shape)


def block_wise_mask(W: np.ndarray, dtype: str, density: float, bh: int = 32, bw: int = 32) -> np.ndarray:
    """Keep the floor(#blocks * density) bh x bw blocks with the largest sum of |w|.

    Ties go to the lower row-major block index.  Sums are exact in float64
    for f16 and int8 inputs; special values rank as in ``vector_wise_mask``."""
    if dtype == "bf16":
        raise ValueError("block-wise scores are exact only for f16 and int8")
    rows, cols = W.shape
    bm, bn = rows // bh, cols // bw
    s = np.abs(decode(W, dtype)).reshape(bm, bh, bn, bw).sum(axis=(1, 3)).reshape(-1)
    keep = int(bm * bn * density)
    order = np.lexsort((np.arange(bm * bn), -s))
    kept = np.zeros(bm * bn, dtype=bool)
    kept[order[:keep]] = True
    return np.repeat(np.repeat(kept.reshape(bm, bn), bh, axis=0), bw, axis=1)


def vector_wise_compress(W: np.ndarray, mask: np.ndarray, v: int = 32):
    """Kept vector indices (ascending, int32) and their values (kept x v)."""
    flat_w = W.reshape(-1, v)
    kept = mask.reshape(-1, v)[:, 0]
    idx = np.nonzero(kept)[0].astype(np.int32)
    return idx, flat_w[idx]


def block_wise_compress(W: np.ndarray, mask: np.ndarray, bh: int = 32, bw: int = 32):
    """Kept block indices (ascending row-major i*bn+j, int32) and their values (kept x bh x bw)."""
    rows, cols = W.shape
    bm, bn = rows // bh, cols // bw
    kept = mask[::bh, ::bw].reshape(-1)
    idx = np.nonzero(kept)[0].astype(np.int32)
    blocks = W.reshape(bm, bh, bn, bw).transpose(0, 2, 1, 3).reshape(bm * bn, bh, bw)
    return idx, blocks[idx]


# --------------------------------------------------------------------------
# tensor-core order of 2:4 metadata
#   Not on the pages: this is the order in which the Blackwell sparse tensor
#   core reads the metadata of a 128-row tile of 16-bit operands, one 32-bit
#   word per row-slot for each 32 columns of the dense operand (one MMA
#   k-step).  Rows are handled in blocks of 16; slot ``16b + 8h + i`` of block
#   ``b`` holds, in its low half, the four codes of row ``16b + i`` for
#   columns ``32s + 16h .. 32s + 16h + 15`` and, in its high half, the same
#   four codes of row ``16b + 8 + i``.  Words are stored k-step by k-step, so
#   that the 128 words of one k-step and one tile are contiguous.  It is the
#   canonical metadata with its 16-bit words permuted, nothing else.
# --------------------------------------------------------------------------
def tc_meta_slot_rows(rows: int) -> int:
    """Slot rows: rows rounded up to a multiple of 128 (whole tensor-core tiles)."""
    return ((rows + 127) // 128) * 128


# Filler for the codes of rows past the matrix: code 0x4 = keep positions 0 and 1.
TC_PAD_CODE_WORD = 0x44444444


def meta_to_tc_layout(meta: np.ndarray, rows: int, cols: int) -> np.ndarray:
    """Canonical 2:4 metadata (rows x ceil(cols/16) uint16) -> tensor-core order.

    Output: uint32 array of shape (cols/32, tc_meta_slot_rows(rows)); codes of
    rows past ``rows`` are the filler 0x4."""
    if cols % 32:
        raise ValueError("tensor-core metadata needs cols % 32 == 0")
    S = cols // 32
    nslots = tc_meta_slot_rows(rows)
    nb = nslots // 16
    canon = np.full((nslots, 2 * S), 0x4444, dtype=np.uint32)
    canon[:rows] = meta[:, : 2 * S].astype(np.uint32)
    C = canon.reshape(nb, 2, 8, S, 2)  # [block][row half][i][s][h]
    word = C[:, 0] | (C[:, 1] << np.uint32(16))  # [block][i][s][h]
    return word.transpose(2, 0, 3, 1).reshape(S, nslots)  # [s][slot 16b + 8h + i]


def meta_from_tc_layout(tc: np.ndarray, rows: int, cols: int) -> np.ndarray:
    """Inverse of ``meta_to_tc_layout`` (canonical rows x ceil(cols/16) uint16)."""
    S = cols // 32
    nslots = tc_meta_slot_rows(rows)
    nb = nslots // 16
    slots = tc.reshape(S, nslots).reshape(S, nb, 2, 8)  # [s][block][h][i]
    word = slots.transpose(1, 3, 0, 2)  # [block][i][s][h]
    lo = word & np.uint32(0xFFFF)
    hi = word >> np.uint32(16)
    canon = np.stack([lo, hi], axis=1).reshape(nslots, 2 * S)[:rows]
    out = np.zeros((rows, meta_words_per_row(cols)), dtype=np.uint16)
    out[:, : 2 * S] = canon.astype(np.uint16)
    return out


# --------------------------------------------------------------------------
# compressed (CSR) form of vector-wise and block-wise masks
#   The kept vectors (blocks) of each row (block row) in ascending column
#   order: an int32 array of row pointers (rows + 1, or block rows + 1)
#   followed by one column index per kept vector (vector column c covers
#   columns v*c .. v*c + v - 1; block column j covers bw*j .. bw*j + bw - 1),
#   and the kept values in the same order.
# --------------------------------------------------------------------------
def vector_wise_csr(W: np.ndarray, mask: np.ndarray, v: int = 32):
    rows, cols = W.shape
    kept = mask.reshape(rows, cols // v, v)[:, :, 0]
    row_ptr = np.concatenate([[0], np.cumsum(kept.sum(axis=1))]).astype(np.int32)
    r_idx, c_idx = np.nonzero(kept)  # row-major order = ascending within each row
    vals = W.reshape(rows, cols // v, v)[r_idx, c_idx]
    return np.concatenate([row_ptr, c_idx.astype(np.int32)]), vals


def block_wise_csr(W: np.ndarray, mask: np.ndarray, bh: int = 32, bw: int = 32):
    rows, cols = W.shape
    bm, bn = rows // bh, cols // bw
    kept = mask[::bh, ::bw]
    row_ptr = np.concatenate([[0], np.cumsum(kept.sum(axis=1))]).astype(np.int32)
    i_idx, j_idx = np.nonzero(kept)
    blocks = W.reshape(bm, bh, bn, bw).transpose(0, 2, 1, 3)[i_idx, j_idx]  # kept x bh x bw
    return np.concatenate([row_ptr, j_idx.astype(np.int32)]), blocks
