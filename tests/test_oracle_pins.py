"""Pins for the CPU oracle: brute force, closed forms, invariants and special cases.

Each test checks the oracle against something other than itself, chosen so
that a plausible slip (a dropped term, a wrong index, a flipped tie-break, a
transposed operand) fails at least one of them.
"""
import itertools
from fractions import Fraction

import numpy as np
import pytest

import oracle as o

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def f16_bits(a):
    return np.asarray(a, dtype=np.float16).view(np.uint16)


def brute_force_mask(vals, n):
    """Lexicographically first n-subset with the largest exact sum of |v| (no NaN)."""
    m = len(vals)
    best, best_s = None, None
    for sub in itertools.combinations(range(m), n):  # lexicographic order
        s = sum(Fraction(abs(float(vals[j]))) for j in sub)
        if best_s is None or s > best_s:
            best, best_s = sub, s
    mask = np.zeros(m, dtype=bool)
    mask[list(best)] = True
    return mask


# ---------------------------------------------------------------- N:M masks
@pytest.mark.parametrize("m", [2, 3, 4, 5, 6, 8])
def test_nm_mask_matches_brute_force(m):
    rng = np.random.default_rng(100 + m)
    # few distinct magnitudes so ties are frequent; both signs and both zeros
    pool = np.array([0.0, -0.0, 0.5, -0.5, 1.0, -1.0, 2.0, -2.0, 3.0], dtype=np.float16)
    W = rng.choice(pool, size=(40, 4 * m)).astype(np.float16)
    for n in range(1, m):
        got = o.nm_mask(W.view(np.uint16), "f16", n, m)
        groups = W.reshape(-1, m)
        want = np.stack([brute_force_mask(g, n) for g in groups]).reshape(W.shape)
        assert (got == want).all(), (m, n)


def test_24_exhaustive_magnitude_grid():
    # every 4-tuple over {0,1,2,3} x {+,-}: 8^4 groups, ties and signed zeros included
    vals = [0.0, -0.0, 1.0, -1.0, 2.0, -2.0, 3.0, -3.0]
    groups = np.array(list(itertools.product(vals, repeat=4)), dtype=np.float16)
    W = groups.reshape(-1, 16)  # 4 groups per row
    bits = W.view(np.uint16)
    pruned, mask = o.nm_prune(bits, "f16", 2, 4)
    want = np.stack([brute_force_mask(g, 2) for g in groups]).reshape(W.shape)
    assert (mask == want).all()
    assert (mask.reshape(-1, 4).sum(axis=1) == 2).all()
    # kept entries keep their exact bits (including -0); dropped slots become +0
    assert (pruned[mask] == bits[mask]).all()
    assert (pruned[~mask] == 0).all()


def test_24_examples_by_hand():
    # (values) -> kept positions, from the definition: two largest |w|, lower position on ties
    cases = {
        (0.5, -3.0, 2.0, 1.0): (1, 2),
        (1.0, 1.0, 1.0, 1.0): (0, 1),
        (0.0, 0.0, 0.0, 7.0): (0, 3),
        (-2.0, 1.0, 2.0, 2.0): (0, 2),
        (0.0, -0.0, 0.0, 0.0): (0, 1),
    }
    for v, keep in cases.items():
        mask = o.nm_mask(f16_bits([v]), "f16", 2, 4)[0]
        assert tuple(np.nonzero(mask)[0]) == keep, v
        vals, meta = o.nm_compress(f16_bits([v * 4]), "f16", 2, 4)  # 16 columns -> one metadata word
        assert int(meta[0, 0]) & 0xF == keep[0] | (keep[1] << 2)


def test_nan_ranks_above_inf():
    v = f16_bits([[1.0, np.inf, np.nan, 2.0]])
    assert tuple(np.nonzero(o.nm_mask(v, "f16", 2, 4)[0])[0]) == (1, 2)
    v = f16_bits([[np.nan, 1.0, np.nan, np.inf]])
    assert tuple(np.nonzero(o.nm_mask(v, "f16", 2, 4)[0])[0]) == (0, 2)
    assert tuple(np.nonzero(o.nm_mask(v, "f16", 1, 4)[0])[0]) == (0,)


def test_int8_magnitude_of_minus_128():
    W = np.array([[-128, 127, 5, -6]], dtype=np.int8)
    assert tuple(np.nonzero(o.nm_mask(W, "i8", 1, 4)[0])[0]) == (0,)
    assert tuple(np.nonzero(o.nm_mask(W, "i8", 2, 4)[0])[0]) == (0, 1)


def test_bf16_decoding_and_ranking():
    x = np.array([1.0, -3.5, 0.0078125, 2.0], dtype=np.float32)
    bits = (x.view(np.uint32) >> 16).astype(np.uint16).reshape(1, 4)
    assert (o.decode(bits, "bf16") == x.astype(np.float64)).all()
    assert tuple(np.nonzero(o.nm_mask(bits, "bf16", 2, 4)[0])[0]) == (1, 3)


@pytest.mark.parametrize("n", [4, 8, 16])
def test_nm_m32_invariants(n):
    rng = np.random.default_rng(n)
    W = (rng.standard_normal((64, 1024)) * 0.02).astype(np.float16)
    W[0, :32] = np.float16(0.01)  # a group of equal magnitudes
    bits = W.view(np.uint16)
    mask = o.nm_mask(bits, "f16", n, 32)
    g_mask = mask.reshape(-1, 32)
    g_mag = np.abs(W.astype(np.float64)).reshape(-1, 32)
    assert (g_mask.sum(axis=1) == n).all()
    kept_min = np.where(g_mask, g_mag, np.inf).min(axis=1)
    drop_max = np.where(~g_mask, g_mag, -np.inf).max(axis=1)
    assert (kept_min >= drop_max).all()
    # boundary ties: the kept entries equal to the threshold are the lowest positions
    for gm, gv in zip(g_mask, g_mag):
        t = gv[gm].min()
        tied = np.nonzero(gv == t)[0]
        kept_tied = np.nonzero(gm & (gv == t))[0]
        assert (kept_tied == tied[: len(kept_tied)]).all()
    assert tuple(np.nonzero(g_mask[0])[0]) == tuple(range(n))


def test_prune_idempotent_and_sparse_input_unchanged():
    rng = np.random.default_rng(7)
    bits = f16_bits(rng.standard_normal((32, 64)))
    p1, _ = o.nm_prune(bits, "f16", 2, 4)
    p2, _ = o.nm_prune(p1, "f16", 2, 4)
    assert (p1 == p2).all()


# ------------------------------------------------------ compress/decompress
@pytest.mark.parametrize("n,m", [(2, 4), (1, 4), (4, 32), (8, 32), (16, 32), (3, 8)])
def test_compress_round_trip(n, m):
    rng = np.random.default_rng(n * 100 + m)
    W = (rng.standard_normal((24, 4 * m)) * 0.02).astype(np.float16)
    W[3, :m] = -0.0
    bits = W.view(np.uint16)
    vals, meta = o.nm_compress(bits, "f16", n, m)
    assert vals.shape == (24, 4 * n)  # n/m of the size (half for 2:4)
    pruned, _ = o.nm_prune(bits, "f16", n, m)
    dec = o.nm_decompress(vals, meta, 24, 4 * m, n, m)
    assert (dec == pruned).all()
    # compressing the pruned matrix again gives the same dense matrix numerically
    v2, m2 = o.nm_compress(pruned, "f16", n, m)
    assert (o.decode(o.nm_decompress(v2, m2, 24, 4 * m, n, m), "f16") == o.decode(pruned, "f16")).all()


def test_compress_transpose_is_compress_of_transpose():
    rng = np.random.default_rng(3)
    bits = f16_bits(rng.standard_normal((32, 48)))
    vT, mT = o.nm_compress(bits, "f16", 2, 4, transpose=True)
    v, m = o.nm_compress(np.ascontiguousarray(bits.T), "f16", 2, 4)
    assert (vT == v).all() and (mT == m).all()


def test_check_counts_violations():
    rng = np.random.default_rng(4)
    bits = f16_bits(rng.standard_normal((16, 32)) + 3.0)  # no zeros
    assert o.nm_check(bits, "f16", 2, 4) == 16 * 8
    pruned, mask = o.nm_prune(bits, "f16", 2, 4)
    assert o.nm_check(pruned, "f16", 2, 4) == 0
    planted = pruned.copy()
    r, c = np.argwhere(~mask)[5]
    planted[r, c] = f16_bits(1.0)
    assert o.nm_check(planted, "f16", 2, 4) == 1
    nan = pruned.copy()
    nan[r, c] = f16_bits(np.nan)
    assert o.nm_check(nan, "f16", 2, 4) == 1
    negz = pruned.copy()
    negz[r, c] = f16_bits(-0.0)
    assert o.nm_check(negz, "f16", 2, 4) == 0


def test_transposable_check_counts_columns_by_hand():
    """cuSPARSELt blog, cusparseLtSpMMAPruneCheck; PyTorch issue #126420 (2:4 in both directions).

    Every row group below holds two nonzeros, so only the column count can flag
    the matrix: column 0 of the first 4-row block holds three nonzeros, column 5
    of the second block holds four, column 2 of the second block holds three."""
    nz = np.array([
        [1, 1, 0, 0, 0, 0, 1, 1],
        [1, 1, 0, 0, 1, 1, 0, 0],
        [1, 0, 1, 0, 0, 0, 1, 1],
        [0, 0, 1, 1, 1, 1, 0, 0],
        [0, 0, 1, 1, 0, 1, 1, 0],
        [1, 0, 1, 0, 0, 1, 0, 1],
        [0, 1, 1, 0, 1, 1, 0, 0],
        [1, 1, 0, 0, 0, 1, 1, 0],
    ], dtype=bool)
    W = f16_bits(np.where(nz, 1.5, 0.0))
    assert o.nm_check(W, "f16", 2, 4) == 0                         # rows conform
    assert o.nm_check(W, "f16", 2, 4, transposable=True) == 3      # three column groups do not
    # rows and columns change roles under transposition
    WT = np.ascontiguousarray(W.T)
    assert o.nm_check(WT, "f16", 2, 4) == 3
    assert o.nm_check(WT, "f16", 2, 4, transposable=True) == 3
    # a violation in a row group and in a column group at once counts twice
    W2 = W.copy()
    W2[0, 2] = f16_bits(2.0)  # row 0's first group gets a third nonzero; column 2, block 0 gets a third
    assert o.nm_check(W2, "f16", 2, 4) == 1
    assert o.nm_check(W2, "f16", 2, 4, transposable=True) == 1 + 4


def test_transposable_nan_scores_as_infinity():
    """A NaN magnitude scores +Inf (the reading that NaN ranks above every number):
    every pattern that keeps a NaN ties at +Inf and the earliest such pattern wins,
    even against patterns that keep much larger finite values."""
    t = np.array([
        [8.0, 8.0, 0.5, np.nan],
        [8.0, 8.0, np.nan, 0.5],
        [1.0, 1.0, 2.0, 2.0],
        [1.0, 1.0, 2.0, 2.0],
    ])
    mask = o.transposable_mask(f16_bits(t), "f16")
    # Canonical order, row 0's pair outermost: row 0 (0,1) with row 1 (0,1) forces rows 2, 3 to
    # (2,3) and keeps no NaN; row 1 (0,2) is next, keeps the NaN at (1, 2), and rows 2, 3
    # complete it as (1,3), (2,3).
    want = np.zeros((4, 4), dtype=bool)
    for r, pair in enumerate(((0, 1), (0, 2), (1, 3), (2, 3))):
        want[r, list(pair)] = True
    assert (mask == want).all()
    # the finite-only optimum (what a NaN scored as 0 would give) keeps the four 8s instead
    finite = np.nan_to_num(t, nan=0.0)
    assert not (o.transposable_mask(f16_bits(finite), "f16") == want).all()
    # bf16 follows the same rule
    bf = (np.asarray(t, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)
    assert (o.transposable_mask(bf, "bf16") == want).all()


# ------------------------------------------------------------ transposable
def test_ninety_patterns_by_bitmask_enumeration():
    count = 0
    for bits in range(1 << 16):
        t = np.array([(bits >> k) & 1 for k in range(16)]).reshape(4, 4)
        if (t.sum(axis=0) == 2).all() and (t.sum(axis=1) == 2).all():
            count += 1
    assert count == 90
    pats = o.transposable_patterns()
    assert len(pats) == 90
    assert len({t.tobytes() for _, t in pats}) == 90
    for _, t in pats:
        assert (t.sum(axis=0) == 2).all() and (t.sum(axis=1) == 2).all()


def _pair_index(row):
    return o.PAIRS.index(tuple(np.nonzero(row)[0]))


def brute_force_transposable(tile):
    """Over all 2^16 masks: valid ones, ordered by their row pairs, first with the max exact score."""
    cands = []
    for bits in range(1 << 16):
        t = np.array([(bits >> k) & 1 for k in range(16)], dtype=bool).reshape(4, 4)
        if (t.sum(axis=0) == 2).all() and (t.sum(axis=1) == 2).all():
            cands.append((tuple(_pair_index(r) for r in t), t))
    cands.sort(key=lambda c: c[0])
    best, best_s = None, None
    for _, t in cands:
        s = sum(Fraction(abs(float(x))) for x in tile[t])
        if best_s is None or s > best_s:
            best, best_s = t, s
    return best


def test_transposable_matches_brute_force():
    rng = np.random.default_rng(11)
    # dyadic magnitudes whose float32 sums are exact, many ties
    pool = np.array([0.0, 0.25, -0.25, 0.5, 1.0, -1.0, 2.0, -3.0], dtype=np.float16)
    W = rng.choice(pool, size=(8, 12)).astype(np.float16)
    mask = o.transposable_mask(W.view(np.uint16), "f16")
    for tr in range(2):
        for tc in range(3):
            tile = W[4 * tr: 4 * tr + 4, 4 * tc: 4 * tc + 4]
            want = brute_force_transposable(tile)
            assert (mask[4 * tr: 4 * tr + 4, 4 * tc: 4 * tc + 4] == want).all(), (tr, tc)


def test_transposable_properties():
    rng = np.random.default_rng(12)
    W = (rng.standard_normal((64, 96)) * 0.05).astype(np.float16)
    bits = W.view(np.uint16)
    pruned, mask, (v, m), (vT, mT) = o.nm_prune_transposable(bits, "f16")
    # 2:4 along rows and along columns of every tile
    assert (mask.reshape(-1, 4).sum(axis=1) == 2).all()
    assert (mask.T.reshape(-1, 4).sum(axis=1) == 2).all()
    assert o.nm_check(pruned, "f16", 2, 4, transposable=True) == 0
    # the row-only greedy optimum bounds the transposable optimum
    mag = np.abs(W.astype(np.float64))
    greedy = o.nm_mask(bits, "f16", 2, 4)
    tile_sum = lambda mk: (mag * mk).reshape(16, 4, 24, 4).sum(axis=(1, 3))
    assert (tile_sum(mask) <= tile_sum(greedy) + 1e-12).all()
    # compressed forms decompress to the pruned matrix and its transpose
    assert (o.nm_decompress(v, m, 64, 96, 2, 4) == pruned).all()
    assert (o.nm_decompress(vT, mT, 96, 64, 2, 4) == pruned.T).all()
    # an already transposable matrix keeps its mask
    again = o.transposable_mask(pruned, "f16")
    nz = o.decode(pruned, "f16") != 0
    assert (again[nz]).all()


def test_transposable_tie_goes_to_earliest_pattern():
    W = np.ones((4, 4), dtype=np.float16).view(np.uint16)
    mask = o.transposable_mask(W, "f16")
    assert (mask == o.transposable_patterns()[0][1]).all()
    # first canonical pattern: rows 0,1 keep (0,1), rows 2,3 keep (2,3)
    assert tuple(np.nonzero(mask[0])[0]) == (0, 1) and tuple(np.nonzero(mask[3])[0]) == (2, 3)


# --------------------------------------------------------------- the product
def test_spmm_matches_exact_rationals():
    rng = np.random.default_rng(21)
    M, K, N = 5, 8, 3
    Wb = f16_bits(rng.standard_normal((M, K)))
    vals, meta = o.nm_compress(Wb, "f16", 2, 4)
    B = rng.standard_normal((K, N)).astype(np.float16).astype(np.float64)
    C = rng.standard_normal((M, N))
    D = o.spmm_compressed(0.5, vals, meta, "f16", M, K, 2, 4, B, beta=-1.25, C=C)
    # exact: sum over the kept entries only, straight from (vals, meta)
    pos = o.meta_positions(meta, M, K, 2, 4)
    v = o.decode(vals, "f16").reshape(M, K // 4, 2)
    for i in range(M):
        for j in range(N):
            acc = Fraction(0)
            for g in range(K // 4):
                for t in range(2):
                    acc += Fraction(v[i, g, t]) * Fraction(B[4 * g + pos[i, g, t], j])
            want = Fraction(0.5) * acc + Fraction(-1.25) * Fraction(C[i, j])
            assert abs(float(want) - D[i, j]) <= 1e-12 * (1 + abs(float(want)))


def test_spmm_special_cases():
    rng = np.random.default_rng(22)
    A = rng.standard_normal((6, 8))
    B = rng.standard_normal((8, 4))
    C = rng.standard_normal((6, 4))
    assert np.array_equal(o.spmm(0.0, A, B, 2.0, C), 2.0 * C)
    nanC = np.full((6, 4), np.nan)
    assert np.isfinite(o.spmm(1.0, A, B, 0.0, nanC)).all()
    assert np.allclose(o.spmm(1.0, A, np.eye(8)), A)
    # orientation: D[i, j] pairs row i of A with column j of B
    assert np.isclose(o.spmm(1.0, A, B)[2, 3], float(np.dot(A[2], B[:, 3])))


def test_spmm_int_exact_and_wrapping():
    rng = np.random.default_rng(23)
    A = rng.integers(-128, 128, size=(4, 64)).astype(np.int8)
    B = rng.integers(-128, 128, size=(64, 3)).astype(np.int8)
    D = o.spmm_int(1, A, B)
    for i in range(4):
        for j in range(3):
            assert int(D[i, j]) == sum(int(A[i, k]) * int(B[k, j]) for k in range(64))
    big = o.spmm_int(2**30, np.full((1, 4), 127, np.int8), np.full((4, 1), 127, np.int8))
    want = (2**30 * 4 * 127 * 127) % 2**32
    want = want - 2**32 if want >= 2**31 else want
    assert int(big[0, 0]) == want
    C = np.array([[7]], dtype=np.int32)
    assert int(o.spmm_int(0, A[:1, :4], B[:4, :1], 3, C)[0, 0]) == 21


def test_masked_weight_grad_by_loops():
    rng = np.random.default_rng(24)
    T, out, inp = 6, 4, 8
    dY = rng.standard_normal((T, out))
    X = rng.standard_normal((T, inp))
    mask = o.transposable_mask(f16_bits(rng.standard_normal((out, inp))), "f16")
    G = o.masked_weight_grad(dY, X, mask)
    for i in range(out):
        for j in range(inp):
            want = sum(dY[t, i] * X[t, j] for t in range(T)) if mask[i, j] else 0.0
            assert abs(G[i, j] - want) <= 1e-12


def test_masked_weight_grad_closed_forms():
    rng = np.random.default_rng(25)
    out, inp = 4, 8
    mask = o.transposable_mask(f16_bits(rng.standard_normal((out, inp))), "f16")
    # X = identity (tokens = input features): the gradient is the masked transpose of dY
    dY = rng.standard_normal((inp, out))
    assert np.array_equal(o.masked_weight_grad(dY, np.eye(inp), mask), np.where(mask, dY.T, 0.0))
    # rank one: dY[t, i] = a_t b_i and X[t, j] = a_t c_j give (sum a_t^2) b_i c_j on kept entries
    a = np.array([1.0, -2.0, 0.5, 3.0, 0.25, -1.0])
    b, c = rng.standard_normal(out), rng.standard_normal(inp)
    G = o.masked_weight_grad(np.outer(a, b), np.outer(a, c), mask)
    want = np.where(mask, (a @ a) * np.outer(b, c), 0.0)
    assert np.allclose(G, want, rtol=1e-13, atol=1e-13)
    assert G.shape == (out, inp)


# ------------------------------------------------- vector- and block-wise masks
def test_vector_wise_literal_score_and_count():
    rng = np.random.default_rng(31)
    W = (rng.standard_normal((8, 64)) * 0.02).astype(np.float16)
    bits = W.view(np.uint16)
    for density in (0.25, 0.5, 0.3):
        mask = o.vector_wise_mask(bits, "f16", density, v=32)
        vec = mask.reshape(-1, 32)
        assert (vec.all(axis=1) | (~vec).all(axis=1)).all()
        assert vec[:, 0].sum() == int(16 * density)
    # brute force: sort by |sum| descending, index ascending
    s = [abs(sum(Fraction(float(x)) for x in vrow)) for vrow in W.reshape(-1, 32)]
    order = sorted(range(16), key=lambda k: (-s[k], k))[:4]
    want = np.zeros(16, bool)
    want[order] = True
    assert (o.vector_wise_mask(bits, "f16", 0.25, 32).reshape(-1, 32)[:, 0] == want).all()
    # the literal score uses the signed sum: +x and -x cancel
    Z = np.zeros((1, 64), np.float16)
    Z[0, :2] = [1.0, -1.0]
    Z[0, 32] = 0.5
    m = o.vector_wise_mask(Z.view(np.uint16), "f16", 0.5, 32)
    assert m[0, 32] and not m[0, 0]
    m2 = o.vector_wise_mask(Z.view(np.uint16), "f16", 0.5, 32, score="sum_of_abs")
    assert m2[0, 0] and not m2[0, 32]


def test_block_wise_brute_force():
    rng = np.random.default_rng(32)
    W = (rng.standard_normal((64, 96)) * 0.02).astype(np.float16)
    bits = W.view(np.uint16)
    mask = o.block_wise_mask(bits, "f16", 0.25, 16, 16)
    assert mask[::16, ::16].sum() == int(4 * 6 * 0.25)
    s = {}
    for i in range(4):
        for j in range(6):
            s[(i, j)] = sum(Fraction(abs(float(x))) for x in W[16 * i:16 * i + 16, 16 * j:16 * j + 16].ravel())
    order = sorted(s, key=lambda ij: (-s[ij], ij[0] * 6 + ij[1]))[:6]
    for (i, j) in s:
        assert mask[16 * i, 16 * j] == ((i, j) in order)
        assert mask[16 * i:16 * i + 16, 16 * j:16 * j + 16].all() == ((i, j) in order)


def test_vw_bw_compress_round_trip():
    rng = np.random.default_rng(33)
    W = (rng.standard_normal((64, 64)) * 0.02).astype(np.float16).view(np.uint16)
    mv = o.vector_wise_mask(W, "f16", 0.25, 32)
    idx, vals = o.vector_wise_compress(W, mv, 32)
    rebuilt = np.zeros(W.size, np.uint16)
    for k, v in zip(idx, vals):
        rebuilt[32 * k: 32 * k + 32] = v
    assert (rebuilt.reshape(W.shape) == np.where(mv, W, 0)).all()
    mb = o.block_wise_mask(W, "f16", 0.25, 32, 32)
    bidx, bvals = o.block_wise_compress(W, mb, 32, 32)
    assert len(bidx) == 1
    i, j = divmod(int(bidx[0]), 2)
    assert (bvals[0] == W[32 * i:32 * i + 32, 32 * j:32 * j + 32]).all()


# ------------------------------------------------ tensor-core metadata order
def test_tc_layout_round_trip_and_grouping():
    rng = np.random.default_rng(41)
    W = f16_bits(rng.standard_normal((40, 96)))
    _, meta = o.nm_compress(W, "f16", 2, 4)
    tc = o.meta_to_tc_layout(meta, 40, 96)
    assert tc.shape == (3, 128)
    assert (o.meta_from_tc_layout(tc, 40, 96) == meta).all()
    # rows 40..47 are the high halves of slots 32..47; slots 48.. are filler
    assert (tc[:, 48:] == o.TC_PAD_CODE_WORD).all()
    assert ((tc[:, 32:48] >> 16) == 0x4444).all()
    # each slot word pairs rows i and i+8 of its 16-row block at the same 16 columns
    for slot in range(40):
        b, j = divmod(slot, 16)
        h, i = divmod(j, 8)
        for s in range(3):
            lo_row, hi_row = 16 * b + i, 16 * b + 8 + i
            assert int(tc[s, slot]) & 0xFFFF == int(meta[lo_row, 2 * s + h])
            if hi_row < 40:
                assert int(tc[s, slot]) >> 16 == int(meta[hi_row, 2 * s + h])


def test_vw_bw_csr_matches_sorted_lists():
    rng = np.random.default_rng(34)
    W = (rng.standard_normal((64, 128)) * 0.02).astype(np.float16).view(np.uint16)
    mv = o.vector_wise_mask(W, "f16", 0.25, 32)
    csr, vals = o.vector_wise_csr(W, mv, 32)
    idx, vals2 = o.vector_wise_compress(W, mv, 32)
    row_ptr, cols_ = csr[:65], csr[65:]
    assert row_ptr[-1] == len(idx) == int(256 * 0.25)
    assert (row_ptr[:-1] * 0 + np.diff(row_ptr) >= 0).all()
    # the CSR order is the ascending global vector order
    assert (np.repeat(np.arange(64), np.diff(row_ptr)) * 4 + cols_ == idx).all()
    assert (vals == vals2).all()
    mb = o.block_wise_mask(W, "f16", 0.25, 32, 32)
    bcsr, blocks = o.block_wise_csr(W, mb, 32, 32)
    bidx, bvals = o.block_wise_compress(W, mb, 32, 32)
    assert (np.repeat(np.arange(2), np.diff(bcsr[:3])) * 4 + bcsr[3:] == bidx).all()
    assert (blocks == bvals).all()


def test_vw_bw_special_values_rank():
    # float64 ordering read for the unspecified cases: Inf above every number,
    # NaN below every number (0 included); ties by the lower index.
    Z = np.zeros((1, 6 * 32), np.float16)
    Z[0, 0] = np.nan                       # vector 0: NaN
    Z[0, 32] = np.inf                      # vector 1: +Inf
    Z[0, 64], Z[0, 65] = np.inf, -np.inf   # vector 2: +Inf + -Inf = NaN (signed sum) / Inf (sum of |w|)
    Z[0, 96] = 1.0                         # vector 3: 1
    Z[0, 128] = -np.inf                    # vector 4: |-Inf| = Inf
    # vector 5: all zeros, score 0
    bits = Z.view(np.uint16)
    kept = lambda m: list(np.nonzero(m.reshape(-1, 32)[:, 0])[0])
    assert kept(o.vector_wise_mask(bits, "f16", 3 / 6, 32)) == [1, 3, 4]
    assert kept(o.vector_wise_mask(bits, "f16", 4 / 6, 32)) == [1, 3, 4, 5]
    assert kept(o.vector_wise_mask(bits, "f16", 5 / 6, 32)) == [0, 1, 3, 4, 5]
    assert kept(o.vector_wise_mask(bits, "f16", 3 / 6, 32, score="sum_of_abs")) == [1, 2, 4]
    B = np.zeros((2, 4), np.float16)
    B[0, 0] = np.nan
    B[1, 3] = np.inf
    mb = o.block_wise_mask(B.view(np.uint16), "f16", 2 / 4, 1, 2)
    assert list(np.nonzero(mb[:, ::2].reshape(-1))[0]) == [1, 3]  # zero block 1 beats the NaN block 0


def test_vw_int8_scores():
    W = np.zeros((1, 96), np.int8)
    W[0, 0], W[0, 1] = -128, 127           # signed sum -1, sum of |w| 255
    W[0, 32] = 100                         # 100
    W[0, 64:66] = -60                      # -120 -> 120
    kept = lambda m: list(np.nonzero(m.reshape(-1, 32)[:, 0])[0])
    assert kept(o.vector_wise_mask(W, "i8", 1 / 3, 32)) == [2]
    assert kept(o.vector_wise_mask(W, "i8", 1 / 3, 32, score="sum_of_abs")) == [0]


# ------------------------------------------------------- storage formats
# The header's storage rules, written out by hand for small rows: bit c % 32 of word
# c / 32 is element c; a 2:4 group g of a row is the 4-bit code i0 | i1 << 2 at bits
# 4 * (g % 4) of uint16 word g / 4; n:m metadata is one uint8 position per kept value.
def test_mask_bits_layout_by_hand():
    mask = np.zeros((2, 70), dtype=bool)
    mask[0, [0, 5, 31, 32, 63, 64]] = True
    mask[1, [1, 69]] = True
    bits = o.mask_to_bits(mask)
    assert bits.shape == (2, 3) and bits.dtype == np.uint32
    assert bits[0].tolist() == [0x80000021, 0x80000001, 0x00000001]
    assert bits[1].tolist() == [0x00000002, 0x00000000, 0x00000020]
    assert (o.bits_to_mask(bits, 70) == mask).all()


def test_canonical_24_metadata_by_hand():
    row = np.arange(20, dtype=np.uint16) + 100  # five groups of four
    keep = [(1, 3), (0, 2), (0, 1), (2, 3), (1, 2)]
    mask = np.zeros((1, 20), dtype=bool)
    for g, (a, b) in enumerate(keep):
        mask[0, [4 * g + a, 4 * g + b]] = True
    vals, meta = o.compress_by_mask(row[None, :], mask, 2, 4)
    assert vals[0].tolist() == [101, 103, 104, 106, 108, 109, 114, 115, 117, 118]
    # codes 0xD, 0x8, 0x4, 0xE in word 0 (groups 0..3), 0x9 in word 1 (group 4)
    assert meta.dtype == np.uint16 and meta[0].tolist() == [0xE48D, 0x0009]
    assert o.meta_words_per_row(20) == 2 and o.meta_words_per_row(16) == 1 and o.meta_words_per_row(4) == 1


def test_nm_position_metadata_by_hand():
    row = np.arange(16, dtype=np.uint16)  # two groups of eight, three kept in each
    mask = np.zeros((1, 16), dtype=bool)
    mask[0, [7, 2, 5]] = True
    mask[0, [8, 9, 15]] = True
    vals, meta = o.compress_by_mask(row[None, :], mask, 3, 8)
    assert vals[0].tolist() == [2, 5, 7, 8, 9, 15]  # ascending position order
    assert meta.dtype == np.uint8 and meta[0].tolist() == [2, 5, 7, 0, 1, 7]


def test_tc_slot_rows_are_whole_tiles():
    assert [o.tc_meta_slot_rows(r) for r in (1, 127, 128, 129, 256, 300)] == [128, 128, 128, 256, 256, 384]


# ------------------------------------------------------ fused SGD re-prune
def bf16_bits(a):
    """float32 values (exactly representable in bf16) as bf16 bit patterns."""
    return (np.asarray(a, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)


def test_sgd_update_hand_cases_f16():
    # exact: 1 - 0.5 * 1 = 0.5; 3 - 2 * 0.25 = 2.5; -2 - 0.25 * (-8) = 0
    got1 = o.decode(o.sgd_update(f16_bits([[1.0]]), f16_bits([[1.0]]), 0.5, "f16"), "f16")
    assert got1[0, 0] == 0.5
    got2 = o.decode(o.sgd_update(f16_bits([[3.0]]), f16_bits([[0.25]]), 2.0, "f16"), "f16")
    assert got2[0, 0] == 2.5
    got3 = o.decode(o.sgd_update(f16_bits([[-2.0]]), f16_bits([[-8.0]]), 0.25, "f16"), "f16")
    assert got3[0, 0] == 0.0
    # rounding to nearest even in f16 (spacing 2**-11 just below 1.0):
    # 1 - 2**-11 is representable; 1 - 2**-12 lies halfway between 1 - 2**-11 (odd) and 1.0 (even) -> 1.0;
    # 1 - 3 * 2**-13 is nearer 1 - 2**-11
    one = f16_bits([[1.0, 1.0, 1.0]])
    g = f16_bits([[2.0 ** -11, 2.0 ** -12, 3 * 2.0 ** -13]])
    got = o.decode(o.sgd_update(one, g, 1.0, "f16"), "f16")[0]
    assert got.tolist() == [1.0 - 2.0 ** -11, 1.0, 1.0 - 2.0 ** -11]


def test_sgd_update_hand_cases_bf16():
    # bf16 spacing just below 1.0 is 2**-8: 1 - 2**-9 is a tie -> 1.0 (even); 1 - 3 * 2**-10 -> 1 - 2**-8
    one = bf16_bits([[1.0, 1.0, 1.0, 4.0]])
    g = bf16_bits([[2.0 ** -9, 3 * 2.0 ** -10, 2.0 ** -8, 1.0]])
    got = o.decode(o.sgd_update(one, g, 1.0, "bf16"), "bf16")[0]
    assert got.tolist() == [1.0, 1.0 - 2.0 ** -8, 1.0 - 2.0 ** -8, 3.0]


def test_sgd_update_rounds_the_product_to_float32_first():
    # lr = 0.1 is not a float32 value: -lr rounds to -0.100000001490116..., and the product with g = 3
    # rounds to float32 before the sum; the result differs from the exactly rounded w - 0.3 in f16
    # only through those roundings, which the float32 path reproduces: w = 1 gives 0.7 -> f16 0.7001953125
    got = o.decode(o.sgd_update(f16_bits([[1.0]]), f16_bits([[3.0]]), 0.1, "f16"), "f16")[0, 0]
    nlr = -np.float32(0.1)
    assert np.float32(nlr * np.float32(3.0)) == np.float32(-0.3)  # the product rounds to the float32 nearest -0.3
    assert got == float(np.float16(np.float32(1.0) + np.float32(-0.3)))
    assert got == 0.7001953125


def test_sgd_update_identities_and_composition():
    rng = np.random.default_rng(41)
    W = f16_bits(rng.standard_normal((16, 32)) * 0.05 + 0.01)  # no -0
    G = f16_bits(rng.standard_normal((16, 32)))
    assert (o.sgd_update(W, G, 0.0, "f16") == W).all()                     # lr = 0
    assert (o.sgd_update(W, f16_bits(np.zeros((16, 32))), 0.3, "f16") == W).all()  # zero gradient
    W_new, pruned, mask, (v, m), (vT, mT) = o.sgd_prune_transposable(W, G, 0.01, "f16")
    # the prune is that of the updated weight, and it is 2:4 in both directions
    p2, mask2, (v2, m2), (vT2, mT2) = o.nm_prune_transposable(W_new, "f16")
    assert (mask == mask2).all() and (v == v2).all() and (vT == vT2).all() and (pruned == p2).all()
    assert o.nm_check(pruned, "f16", 2, 4, transposable=True) == 0
    # elementwise: the update is w - lr * g up to the two float32 roundings and the final f16 rounding
    w, gg, wn = o.decode(W, "f16"), o.decode(G, "f16"), o.decode(W_new, "f16")
    assert np.abs(wn - (w - 0.01 * gg)).max() <= np.abs(w - 0.01 * gg).max() * 2.0 ** -10


def test_int8_output_scale_round_and_saturate():
    A = np.array([[1, 2, 0, 0], [127, 127, 0, 0], [-128, -128, 0, 0]], dtype=np.int8)
    B = np.array([[1, 3], [1, -1], [5, 5], [7, 7]], dtype=np.int8)
    # acc = [[3, 1], [254, 254], [-256, -256]]
    assert (A.astype(np.int64) @ B.astype(np.int64)).tolist() == [[3, 1], [254, 254], [-256, -256]]
    got = o.spmm_int8_out(0.5, A, B)
    # 1.5 -> 2 and 0.5 -> 0 (ties to even); 127 stays; -128 saturates from -128 exactly
    assert got.tolist() == [[2, 0], [127, 127], [-128, -128]]
    got = o.spmm_int8_out(1.0, A, B)
    assert got.tolist() == [[3, 1], [127, 127], [-128, -128]]  # saturation both ways
    C = np.array([[10, -10], [0, 0], [100, 100]], dtype=np.int8)
    got = o.spmm_int8_out(0.25, A, B, beta=0.5, C=C)
    # 0.75 + 5 = 5.75 -> 6; 0.25 - 5 = -4.75 -> -5; 63.5 -> 64 (tie to even); -64 + 50 = -14
    assert got.tolist() == [[6, -5], [64, 64], [-14, -14]]
    # above 2**24 the int32 -> float32 conversion rounds to even: 127 * 127 * 1041 = 16790289 -> 16790288,
    # and 16790288 * 2**-19 = 32.0250244... -> 32
    A2 = np.full((1, 1041), 127, dtype=np.int8)
    B2 = np.full((1041, 1), 127, dtype=np.int8)
    assert float(np.float32(127 * 127 * 1041)) == 16790288.0
    assert o.spmm_int8_out(2.0 ** -19, A2, B2)[0, 0] == 32
