"""Pins of the CPU oracle against facts fixed by the hc_fused page and by arithmetic.

Each test uses inputs whose correct result is known in closed form (or by exact
rational arithmetic), chosen so that a plausible slip in the oracle -- a wrong
summation order, a dropped reset, a transposed operand, a wrong group index --
changes the result.  None of them re-types the oracle's own loops.
"""
from fractions import Fraction

import numpy as np
import pytest

import hcmix_inputs as hi
import oracle
from pin_inputs import rms_pin_closed_form, rms_pin_inputs

F32 = np.float32
TWO24 = 2.0 ** 24


def bf16(vals):
    return hi.bf16_bits_from_f64(np.asarray(vals, np.float64))


def f32_round_exact(q: Fraction) -> np.float32:
    """Correctly rounded (nearest, ties to even) fp32 of an exact rational."""
    c = np.float32(float(q))
    best = None
    for cand in (np.nextafter(c, F32(-np.inf)), c, np.nextafter(c, F32(np.inf))):
        dist = abs(Fraction(float(cand)) - q)
        key = (dist, int(np.asarray(cand).view(np.uint32)) & 1)
        if best is None or key < best[0]:
            best = (key, cand)
    return F32(best[1])


# ---------------------------------------------------------------- exactness facts

def test_bf16_values_are_exact_in_tf32():
    """Every bf16 value fits tf32 without rounding (page docstring, tf32x3 bullet).

    Round every finite bf16 to a 10-bit mantissa (round to nearest, ties away, as
    cvt.rna.tf32.f32 does) and check nothing changes.
    """
    bits = np.arange(1 << 16, dtype=np.uint32)
    f = (bits << 16).view(np.float32)
    finite = np.isfinite(f)
    u = f[finite].view(np.uint32).astype(np.uint64)
    rna = ((u + np.uint64(1 << 12)) & ~np.uint64((1 << 13) - 1)).astype(np.uint32)
    assert np.array_equal(rna, u.astype(np.uint32))


def test_bf16_squares_are_exact_in_fp32():
    """x*x for every bf16 with |x| < 2**63 is exact in fp32 (8-bit significand squared)."""
    bits = np.arange(1 << 16, dtype=np.uint32)
    f = (bits << 16).view(np.float32)
    keep = np.isfinite(f) & (np.abs(f) < 2.0 ** 63) & ((np.abs(f) >= 2.0 ** -63) | (f == 0))
    f = f[keep]
    assert np.array_equal((f * f).astype(np.float64), f.astype(np.float64) ** 2)


# ---------------------------------------------------------------- chunk dot

def test_chunk_dot_is_correctly_rounded_exact_dot():
    """Brute force: on random 64-term chunks the oracle's chunk dot equals the
    exact rational dot product rounded once to fp32."""
    rng = np.random.default_rng(11)
    for trial in range(60):
        xb = bf16(rng.standard_normal(64) * (8.0 if trial % 3 == 0 else 1.0))
        w = (rng.standard_normal(64) * 0.007).astype(np.float32)
        xs = hi.bf16_bits_to_f32(xb)
        exact = sum(Fraction(float(a)) * Fraction(float(b)) for a, b in zip(xs, w))
        assert oracle.chunk_dot(xb, w) == f32_round_exact(exact)


def test_chunk_dot_rounds_once():
    """Terms 2**24, 1, 1: the exact sum 2**24+2 is an fp32 value; rounding after
    every add would lose both ones (2**24+1 ties to 2**24)."""
    xb = bf16([2.0 ** 12, 1.0, 1.0] + [0.0] * 61)
    w = np.array([2.0 ** 12, 1.0, 1.0] + [0.0] * 61, np.float32)
    assert oracle.chunk_dot(xb, w) == F32(TWO24 + 2)
    assert oracle.chunk_dot_seq_f32(xb, w) == F32(TWO24)


# ---------------------------------------------------------------- slice / total order

def _stats_with_chunk_values(values):
    """x, W over K = 64*len(values) whose chunk dots for output 0 are `values`
    (each an exact power of two or zero), other outputs zero."""
    n = len(values)
    K = 64 * n
    x = np.zeros((1, K), np.float64)
    W = np.zeros((24, K), np.float32)
    for c, v in enumerate(values):
        if v == 0:
            continue
        e = int(np.log2(v))
        a = 2.0 ** (e // 2)
        x[0, 64 * c] = a
        W[0, 64 * c] = v / a
    return oracle.stats(bf16(x), W)


def test_slice_totals_added_in_slice_order_from_zero():
    """Slice 0 holds one chunk of 2**24, every later slice one chunk of 1.

    Forward order from zero: each +1 ties back to 2**24, so mix = 2**24.
    Reverse or pairwise order would first collect the ones and give 2**24 + 80.
    """
    vals = []
    for s in range(80):
        vals += [TWO24 if s == 0 else 1.0, 0.0, 0.0, 0.0]
    mix, _ = _stats_with_chunk_values(vals)
    assert mix[0, 0] == F32(TWO24)


def test_chunks_added_in_order_within_slice():
    """Chunk dots (2**24, 1, 1, 1): each +1 ties back to 2**24, so mix = 2**24.
    Adding the chunks in reverse would give 3 + 2**24 -> 2**24 + 4."""
    mix, _ = _stats_with_chunk_values([TWO24, 1.0, 1.0, 1.0])
    assert mix[0, 0] == F32(TWO24)
    mix, _ = _stats_with_chunk_values([1.0, 1.0, 1.0, TWO24])
    assert mix[0, 0] == F32(TWO24 + 4)


def test_slice_accumulator_restarts_at_zero():
    """Slice 0 chunks (2**24, 0, 0, 0), slice 1 chunks (1, 1, 1, 1): slice 1's
    total restarts at zero (4), so mix = 2**24 + 4; carrying the slice-0 value
    over would double the large term."""
    mix, _ = _stats_with_chunk_values([TWO24, 0.0, 0.0, 0.0, 1.0, 1.0, 1.0, 1.0])
    assert mix[0, 0] == F32(TWO24 + 4)


def test_sq_tree_bit_order():
    """Squares 2**24 at k=0 and 1 at k=1 and k=3.  The page's tree joins bit 1
    before bit 0, so the two ones meet first: 2**24 + 2.  A running sum or a
    tree starting with bit 0 rounds each one away: 2**24."""
    x = np.zeros(64)
    x[0], x[1], x[3] = 2.0 ** 12, 1.0, 1.0
    assert oracle.sq_tree(bf16(x)) == F32(TWO24 + 2)


def test_sq_tree_halves_last():
    """Squares 2**24 at k=0, 1 at k=32 and k=33: the halves meet last, after the
    two ones have formed 2, giving 2**24 + 2 (halves first would give 2**24)."""
    x = np.zeros(64)
    x[0], x[32], x[33] = 2.0 ** 12, 1.0, 1.0
    assert oracle.sq_tree(bf16(x)) == F32(TWO24 + 2)


def test_sq_tree_first_level_is_bit4():
    """Squares 2**24 at k=0 and 1 at k=16 and k=17: bit 4 pairs (0,16) and (1,17)
    first: 2**24+1 ties to 2**24 and 0+1 = 1; bits 3, 2, 1 add zeros; bit 0 then
    gives 2**24 + 1 -> 2**24 again.  So the tree yields 2**24, whereas a tree
    whose first level is bit 0 pairs (16,17) into 2 and yields 2**24 + 2."""
    x = np.zeros(64)
    x[0], x[16], x[17] = 2.0 ** 12, 1.0, 1.0
    assert oracle.sq_tree(bf16(x)) == F32(TWO24)


def test_sq_of_ones_is_k():
    for K in (256, 1024, 20480):
        x = bf16(np.ones((2, K)))
        _, sq = oracle.stats(x, np.zeros((24, K), np.float32))
        assert np.all(sq == F32(K))


# ---------------------------------------------------------------- layout and indexing

def test_integer_inputs_exact_any_order():
    """x in {-4..4}, W in {-8..8}: every partial sum is an integer below 2**24,
    so mix equals the exact integer product x @ W.T bit for bit."""
    rng = np.random.default_rng(5)
    for K in (256, 1024):
        xi = rng.integers(-4, 5, size=(7, K))
        wi = rng.integers(-8, 9, size=(24, K))
        mix, sq = oracle.stats(bf16(xi), wi.astype(np.float32))
        assert np.array_equal(mix.astype(np.int64), xi @ wi.T)
        assert np.array_equal(sq.astype(np.int64), (xi * xi).sum(1))


def test_one_hot_row_selects_weight_column():
    K = 512
    W = (np.random.default_rng(3).standard_normal((24, K)) * 0.01).astype(np.float32)
    for k in (0, 63, 64, 255, 256, 511):
        x = np.zeros((1, K)); x[0, k] = 1.0
        mix, sq = oracle.stats(bf16(x), W)
        assert np.array_equal(mix[0], W[:, k]) and sq[0] == 1.0


def test_row_stride_is_honoured():
    K = 512
    rng = np.random.default_rng(8)
    xs = bf16(rng.standard_normal((5, K + 64)))
    W = (rng.standard_normal((24, K)) * 0.05).astype(np.float32)
    Wpad = np.zeros((24, K + 32), np.float32); Wpad[:, :K] = W
    a = oracle.stats(xs[:, :K], Wpad[:, :K], K=K)
    b = oracle.stats(np.ascontiguousarray(xs[:, :K]), W)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


# ---------------------------------------------------------------- against double precision

def test_slice_order_equals_unsplit_sum_when_exact():
    """Ordered slice sum == unsplit sum in fp64 when every product and partial sum
    is exact in double: W on a 2**-12 grid within [-1, 1), x bf16 in [-4, 4)."""
    rng = np.random.default_rng(9)
    K = 1024
    x = bf16(np.clip(rng.standard_normal((4, K)), -3.9, 3.9))
    W = (np.round(rng.uniform(-1, 1, (24, K)) * 4096) / 4096).astype(np.float32)
    m64, _ = oracle.stats_f64(x, W)
    u64 = oracle.mix_unsplit_f64(x, W)
    assert np.array_equal(m64, u64)


def test_fp32_oracle_close_to_fp64_on_workload():
    x = hi.make_x(8)
    W = hi.make_w()
    mix, sq = oracle.stats(x, W)
    m64, s64 = oracle.stats_f64(x, W)
    u64 = oracle.mix_unsplit_f64(x, W)
    assert np.max(np.abs(m64 - u64)) < 1e-12
    assert np.max(np.abs(mix - m64)) < 3e-6
    assert np.max(np.abs(sq - s64) / s64) < 1e-6


def test_brute_force_tiny_stats_match_exact_rational_structure():
    """Tiny K=256 rows: rebuild each chunk dot as an exact rational rounded once,
    then the fp32 slice adds, and compare with the oracle bit for bit."""
    rng = np.random.default_rng(12)
    K = 512
    x = bf16(rng.standard_normal((2, K)))
    W = (rng.standard_normal((3, K)) * 0.05).astype(np.float32)
    mix, _ = oracle.stats(x, W)
    xf = hi.bf16_bits_to_f32(x)
    for m in range(2):
        for j in range(3):
            tot = F32(0)
            for s in range(K // 256):
                acc = F32(0)
                for c in range(4):
                    k0 = 256 * s + 64 * c
                    q = sum(Fraction(float(xf[m, k])) * Fraction(float(W[j, k]))
                            for k in range(k0, k0 + 64))
                    acc = F32(acc + f32_round_exact(q))
                tot = F32(tot + acc)
            assert mix[m, j] == tot


# ---------------------------------------------------------------- epilogue

def test_zero_weights_give_half_one_quarter():
    K = 1024
    x = bf16(np.random.default_rng(1).standard_normal((3, K)))
    W = np.zeros((24, K), np.float32)
    pre, post, comb, _, _ = oracle.fused(x, W, hi.make_scale(), np.zeros(24, np.float32))
    assert np.all(pre == F32(0.5)) and np.all(post == F32(1.0)) and np.all(comb == F32(0.25))


def test_zero_activation_gives_logits_equal_base():
    """x = 0: sq = 0, r = 1/sqrt(rms_eps) (finite), mix*r = 0, so logit = base."""
    K = 512
    x = bf16(np.zeros((1, K)))
    W = hi.make_w(K=K)
    base = hi.make_base()
    pre, post, comb, mix, sq = oracle.fused(x, W, hi.make_scale(), base, iters=0)
    b = base.astype(np.float64)
    assert sq[0] == 0 and np.all(mix == 0)
    np.testing.assert_allclose(pre[0], 1 / (1 + np.exp(-b[:4])), rtol=0, atol=2e-7)
    np.testing.assert_allclose(post[0], 2 / (1 + np.exp(-b[4:8])), rtol=0, atol=4e-7)
    np.testing.assert_allclose(comb[0].reshape(-1), np.exp(b[8:]), rtol=3e-7)


def test_epilogue_groups_and_comb_layout():
    """K = 1024, x = 1, rms_eps = 0: sq = K, 1/K exact, so r = 1 exactly.
    W[j, :] = c_j / K gives mix_j = c_j exactly.  With hc_scale = (1, 2, 3) the
    logits are c_j * scale[g(j)] + base_j; compare pre/post/comb with the fp64
    closed form (comb row-major, rows normalised first)."""
    K = 1024
    c = (np.arange(24) - 11.5) / 8.0
    W = np.repeat((c / K)[:, None], K, axis=1).astype(np.float32)
    x = bf16(np.ones((1, K)))
    scale = np.array([1.0, 2.0, 3.0], np.float32)
    base = (np.arange(24) * 0.03 - 0.2).astype(np.float32)
    # a non-separable comb block, so Sinkhorn's answer is not uniform
    base[8:] += np.array([0.9, -0.4, 0.0, 0.3, -0.8, 0.5, 0.1, -0.2,
                          0.4, 0.0, -0.6, 0.7, -0.1, 0.2, 0.6, -0.5], np.float32)
    pre, post, comb, mix, sq = oracle.fused(x, W, scale, base, iters=20, rms_eps=0.0)
    assert np.array_equal(mix[0], c.astype(np.float32)) and sq[0] == K
    g = np.array([0] * 4 + [1] * 4 + [2] * 16)
    logit = c * np.array([1.0, 2.0, 3.0])[g] + base.astype(np.float64)
    np.testing.assert_allclose(pre[0], 1 / (1 + np.exp(-logit[:4])), atol=3e-7)
    np.testing.assert_allclose(post[0], 2 / (1 + np.exp(-logit[4:8])), atol=5e-7)
    C = np.exp(logit[8:]).reshape(4, 4)
    for _ in range(20):
        C = C / C.sum(1, keepdims=True)
        C = C / C.sum(0, keepdims=True)
    np.testing.assert_allclose(comb[0], C, atol=2e-6)
    # the transposed layout is a different matrix: the check above must see it
    assert np.max(np.abs(C - C.T)) > 1e-3


def test_sinkhorn_uniform_and_rank_one():
    one = oracle.sinkhorn(np.ones((4, 4)), 20)
    assert np.all(one == F32(0.25))
    a = np.array([0.3, -1.0, 2.0, 0.5]); b = np.array([1.0, 0.2, -0.7, 0.0])
    C = np.exp(a[:, None] + b[None, :]).astype(np.float32)
    out = oracle.sinkhorn(C, 1)
    np.testing.assert_allclose(out, 0.25, rtol=0, atol=4 * 2 ** -24)


def test_sinkhorn_invariants_and_permutation():
    rng = np.random.default_rng(4)
    for _ in range(50):
        L = rng.standard_normal((4, 4)) * 0.8
        C = oracle.sinkhorn(np.exp(L).astype(np.float32), 20)
        assert np.all(C > 0)
        np.testing.assert_allclose(C.sum(0), 1.0, atol=4 * 2 ** -23)
        np.testing.assert_allclose(C.sum(1), 1.0, atol=1e-5)
        p, q = rng.permutation(4), rng.permutation(4)
        Cp = oracle.sinkhorn(np.exp(L[p][:, q]).astype(np.float32), 20)
        np.testing.assert_allclose(Cp, C[p][:, q], atol=1e-6)


def test_sinkhorn_zero_iterations_is_exp():
    L = np.linspace(-1, 1, 16).astype(np.float32)
    mix = np.zeros((1, 24), np.float32)
    base = np.concatenate([np.zeros(8, np.float32), L])
    _, _, comb = oracle.epilogue(mix, np.zeros(1, np.float32), 1024, np.ones(3, np.float32),
                                 base, iters=0)
    np.testing.assert_allclose(comb[0].reshape(-1), np.exp(L.astype(np.float64)), rtol=2.5e-7)


def test_hc_eps_enters_every_normalisation():
    """All-equal logits with hc_eps = e: each row sum is 4 and each column sum
    4/(4+e) * ..., so after one round of rows then columns every entry is
    (1/(4+e)) / (4/(4+e) + e)."""
    e = 0.5
    C = oracle.sinkhorn(np.ones((4, 4), np.float32), 1, e)
    r = 1.0 / (4.0 + e)
    np.testing.assert_allclose(C, r / (4 * r + e), rtol=1e-6)


def test_fp32_epilogue_close_to_fp64():
    x = hi.make_x(16)
    W = hi.make_w()
    sc, bs = hi.make_scale(), hi.make_base()
    pre, post, comb, mix, sq = oracle.fused(x, W, sc, bs)
    p64, q64, c64 = oracle.epilogue_f64(mix, sq, x.shape[1], sc, bs)
    assert np.max(np.abs(pre - p64)) < 1e-6
    assert np.max(np.abs(post - q64)) < 2e-6
    assert np.max(np.abs(comb - c64)) < 2e-6
    # columns are normalised last, so they sum to 1 up to rounding
    np.testing.assert_allclose(comb.sum(1), 1.0, atol=4 * 2 ** -23)
    # rows: 20 rounds do not always converge to 1e-5 on this distribution; the
    # deviation is the iteration's, so fp64 Sinkhorn of the same logits shows it too
    np.testing.assert_allclose(comb.sum(2), c64.sum(2), atol=1e-6)


def test_sinkhorn_rows_converge_on_moderate_logits():
    rng = np.random.default_rng(21)
    for _ in range(200):
        C = oracle.sinkhorn(np.exp(rng.uniform(-1, 1, (4, 4))).astype(np.float32), 20)
        np.testing.assert_allclose(C.sum(1), 1.0, atol=1e-5)
        np.testing.assert_allclose(C.sum(0), 1.0, atol=4 * 2 ** -23)


# ---------------------------------------------------------------- rms placement

@pytest.mark.parametrize("case", ["one_hot", "all_ones"])
def test_rms_eps_inside_the_root_and_one_over_k(case):
    """r = 1/sqrt(sq * (1/K) + rms_eps): on these inputs r is exact, so the
    oracle's logits equal the closed form to rounding, and each plausible
    misreading (eps outside the root, eps after the reciprocal, no 1/K) moves
    mix * r, hence the outputs, far outside the epilogue tolerance."""
    x, W, eps, r, c = rms_pin_inputs(case)
    K = x.shape[1]
    scale = np.array([1.0, 2.0, 3.0], np.float32)
    base = (np.arange(24) * 0.03 - 0.2).astype(np.float32)
    pre, post, comb, mix, sq = oracle.fused(x, W, scale, base, iters=20, rms_eps=eps)
    assert np.array_equal(mix[0].astype(np.float64) * r, c)
    p, q, C = rms_pin_closed_form(c, scale, base)
    np.testing.assert_allclose(pre[0], p, atol=3e-7)
    np.testing.assert_allclose(post[0], q, atol=5e-7)
    np.testing.assert_allclose(comb[0], C, atol=2e-6)
    s = float(sq[0]) / K
    mix64 = mix[0].astype(np.float64)
    for wrong_r in (1 / (np.sqrt(s) + eps), 1 / np.sqrt(s) + eps, 1 / np.sqrt(float(sq[0]) + eps)):
        pw, qw, Cw = rms_pin_closed_form(mix64 * wrong_r, scale, base)
        worst = max(np.abs(pw - p).max(), np.abs(qw - q).max(), np.abs(Cw - C).max())
        assert worst > 1e-3, f"misreading r = {wrong_r} would go unnoticed"
