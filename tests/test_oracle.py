"""Pins for the CPU oracle (D = A * B^T, fp64 sums, one bf16 rounding).

None of these compare the oracle with itself: each checks it against something
the definition or mathematics fixes independently -- exact rational brute force,
hand-derived rounding cases, closed forms (identity, permutation, all-ones,
integer inputs), an fp64 library matmul, and the library's own fp32 -> bf16
rounding.  A dropped term, a wrong sign, index or stride, a transposed operand,
or a rounding done in the wrong precision fails at least one of them.
"""
from __future__ import annotations

import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from warp_specialized_tma_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "bf16_rne_cases.txt")


# ---------------------------------------------------------------------------
# An independent rounding: exact rationals, nearest, ties to even onto bf16.
# ---------------------------------------------------------------------------
def exact_rne_bf16(x: Fraction, negative_zero: bool = False) -> int:
    if x == 0:
        return 0x8000 if negative_zero else 0x0000
    sign = 0x8000 if x < 0 else 0
    a = abs(x)
    # E with 2^E <= a < 2^(E+1)
    E = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** E > a:
        E -= 1
    while Fraction(2) ** (E + 1) <= a:
        E += 1
    grid = E - 7 if E >= -126 else -133
    q = a / Fraction(2) ** grid
    fl = q.numerator // q.denominator
    rem = q - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    if grid == -133:
        return sign | fl
    if fl == 256:
        fl, E = 128, E + 1
    if E > 127:
        return sign | 0x7F80
    return sign | ((E + 127) << 7) | (fl - 128)


def bf16_value(bits: int) -> Fraction:
    """Exact value of a finite bf16 pattern."""
    s = -1 if bits & 0x8000 else 1
    e = (bits >> 7) & 0xFF
    f = bits & 0x7F
    if e == 0:
        return s * Fraction(f) * Fraction(2) ** -133
    return s * Fraction(128 + f) * Fraction(2) ** (e - 127 - 7)


def random_bf16_bits(rng: np.random.Generator, shape, lo_exp=-6, hi_exp=6) -> np.ndarray:
    """Random finite bf16 patterns with exponents in [lo_exp, hi_exp]."""
    sign = rng.integers(0, 2, size=shape).astype(np.uint16) << 15
    exp = (rng.integers(lo_exp, hi_exp + 1, size=shape) + 127).astype(np.uint16) << 7
    frac = rng.integers(0, 128, size=shape).astype(np.uint16)
    return (sign | exp | frac).astype(np.uint16)


# ---------------------------------------------------------------------------
# Rounding pins
# ---------------------------------------------------------------------------
def _golden_cases():
    cases = []
    with open(GOLDEN) as fh:
        for line in fh:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            val, want = line.split()
            cases.append((float.fromhex(val), int(want, 16), val))
    return cases


@pytest.mark.parametrize("value,want,text", _golden_cases())
def test_rne_golden_cases(value, want, text):
    got = int(oracle.bf16_from_f64(np.array([value]))[0])
    assert got == want, f"{text}: got {got:#06x}, want {want:#06x}"


def test_golden_cases_agree_with_exact_rational_rounding():
    # the hand-derived table and the rational rounding are independent; both must agree
    for value, want, text in _golden_cases():
        if math.isinf(value):
            continue
        got = exact_rne_bf16(Fraction(value), negative_zero=math.copysign(1.0, value) < 0)
        assert got == want, text


def test_rne_matches_exact_rationals_random():
    rng = np.random.default_rng(11)
    # values spanning normal, subnormal and overflow ranges, plus near-ties
    mant = rng.random(4000) + 1.0
    exps = rng.integers(-140, 130, size=4000)
    vals = np.ldexp(mant, exps) * np.where(rng.random(4000) < 0.5, -1.0, 1.0)
    ties = np.array([float(bf16_value(int(b))) for b in random_bf16_bits(rng, 500, -126, 120)])
    ties = ties * (1.0 + 2.0 ** -8)   # lands near the midpoints of the bf16 grid
    vals = np.concatenate([vals, ties])
    got = oracle.bf16_from_f64(vals)
    for v, g in zip(vals, got):
        want = exact_rne_bf16(Fraction(float(v)))
        assert int(g) == want, (v.hex(), hex(int(g)), hex(want))


def test_rne_matches_library_fp32_rounding():
    # torch rounds fp32 -> bf16 to nearest even; fp32 values are exact in fp64,
    # so a direct fp64 rounding must give the same bits.
    g = torch.Generator().manual_seed(5)
    x = torch.randn(200000, generator=g, dtype=torch.float32) * 3.0
    x = torch.cat([x, torch.randn(20000, generator=g) * 1e-39, torch.randn(20000, generator=g) * 1e30])
    want = x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.bf16_from_f64(x.double().numpy())
    assert np.array_equal(got, want)


def test_widening_all_patterns():
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    wide = oracle.f64_from_bf16(pats)
    lib = torch.from_numpy(pats.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    finite = np.isfinite(lib)
    assert np.array_equal(np.isnan(wide), np.isnan(lib))
    assert np.array_equal(wide[finite], lib[finite])
    # widening then rounding is the identity on every non-NaN pattern
    back = oracle.bf16_from_f64(wide)
    notnan = ~np.isnan(wide)
    assert np.array_equal(back[notnan], pats[notnan])


# ---------------------------------------------------------------------------
# GEMM pins
# ---------------------------------------------------------------------------
def _exact_gemm(Ab, Bb, K):
    M, N = Ab.shape[0], Bb.shape[0]
    Af = [[bf16_value(int(Ab[m, k])) for k in range(K)] for m in range(M)]
    Bf = [[bf16_value(int(Bb[n, k])) for k in range(K)] for n in range(N)]
    return [[sum((Af[m][k] * Bf[n][k] for k in range(K)), Fraction(0)) for n in range(N)]
            for m in range(M)]


@pytest.mark.parametrize("pad", [0, 8])
def test_bruteforce_tiny_shapes_exact(pad):
    rng = np.random.default_rng(100 + pad)
    for M in range(1, 9):
        for N in range(1, 9):
            for K in (1, 2, 3, 5, 8):
                ld = K + pad
                A = random_bf16_bits(rng, (M, ld))
                B = random_bf16_bits(rng, (N, ld))
                ref64, refbf = oracle.gemm_rows(A, B, K=K)
                exact = _exact_gemm(A, B, K)
                for m in range(M):
                    for n in range(N):
                        # <= 8 products of 8-bit significands with exponents in
                        # [-12, 12]: the fp64 sum is exact, so equality is exact.
                        assert Fraction(float(ref64[m, n])) == exact[m][n], (M, N, K, m, n)
                        assert int(refbf[m, n]) == exact_rne_bf16(exact[m][n]), (M, N, K, m, n)


def test_against_fp64_library_matmul_nonsquare():
    # non-square shapes so that a transposed operand cannot pass
    A, B = inputs.make_problem(37, 53, 71, "normal", seed=9)
    Ab, Bb = inputs.bits(A), inputs.bits(B)
    ref64, refbf = oracle.gemm_rows(Ab, Bb)
    A64 = oracle.f64_from_bf16(Ab)
    B64 = oracle.f64_from_bf16(Bb)
    lib = A64 @ B64.T
    bound = 71 * 2.0 ** -52 * (np.abs(A64) @ np.abs(B64).T)
    assert ref64.shape == (37, 53)
    assert np.all(np.abs(ref64 - lib) <= bound)
    assert np.array_equal(refbf, oracle.bf16_from_f64(ref64))


def test_identity_operands_exact():
    g = torch.Generator().manual_seed(3)
    K = 96
    Bm = inputs.make_operand(40, K, None, "normal", g)
    eye = torch.eye(K, dtype=torch.bfloat16)
    # A = I  ->  D[m, n] = B[n, m]
    _, d1 = oracle.gemm_rows(inputs.bits(eye), inputs.bits(Bm))
    assert np.array_equal(d1, inputs.bits(Bm).T)
    # B = I  ->  D = A
    Am = inputs.make_operand(33, K, None, "uniform", g)
    _, d2 = oracle.gemm_rows(inputs.bits(Am), inputs.bits(eye))
    assert np.array_equal(d2, inputs.bits(Am))


def test_permutation_operand_exact():
    g = torch.Generator().manual_seed(4)
    K, N = 64, 48
    perm = torch.randperm(K, generator=g)
    P = torch.zeros((K, K), dtype=torch.bfloat16)
    P[torch.arange(K), perm] = 1.0          # P[m, k] = 1 iff k == perm[m]
    Bm = inputs.make_operand(N, K, None, "normal", g)
    _, d = oracle.gemm_rows(inputs.bits(P), inputs.bits(Bm))
    want = inputs.bits(Bm)[:, perm.numpy()].T   # D[m, n] = B[n, perm[m]]
    assert np.array_equal(d, want)


def test_all_ones_closed_forms():
    g = torch.Generator().manual_seed(6)
    K, N = 257, 19
    Bm = inputs.make_operand(N, K, None, "normal", g)
    ones = torch.ones((5, K), dtype=torch.bfloat16)
    ref64, _ = oracle.gemm_rows(inputs.bits(ones), inputs.bits(Bm))
    B64 = Bm.double().numpy()
    rowsum = np.array([math.fsum(B64[n]) for n in range(N)])
    # every row of D is the vector of row sums of B (exact: the fp64 sum of
    # 257 bf16 values of this range needs far fewer than 53 bits)
    assert np.array_equal(ref64, np.broadcast_to(rowsum, (5, N)))
    # A = B = 1: every entry is K
    r2, b2 = oracle.gemm_rows(inputs.bits(ones), inputs.bits(torch.ones((3, K), dtype=torch.bfloat16)))
    assert np.all(r2 == K)
    assert np.all(b2 == exact_rne_bf16(Fraction(K)))


def test_integer_inputs_exact():
    A, B = inputs.make_problem(29, 31, 300, "int2", seed=8)
    ref64, refbf = oracle.gemm_rows(inputs.bits(A), inputs.bits(B))
    Ai = A.to(torch.int64).numpy()
    Bi = B.to(torch.int64).numpy()
    exact = Ai @ Bi.T
    assert np.array_equal(ref64, exact.astype(np.float64))
    want = np.array([[exact_rne_bf16(Fraction(int(v))) for v in row] for row in exact], dtype=np.uint16)
    assert np.array_equal(refbf, want)


def test_row_subset_and_padding_agree_with_dense():
    A, B = inputs.make_problem(45, 22, 70, "normal", seed=12)
    Ap, Bp = inputs.make_problem(45, 22, 70, "normal", seed=12, lda=88, ldb=72)
    full64, fullbf = oracle.gemm_rows(inputs.bits(A), inputs.bits(B))
    pad64, padbf = oracle.gemm_rows(inputs.bits(Ap), inputs.bits(Bp), K=70)
    assert np.array_equal(full64, pad64) and np.array_equal(fullbf, padbf)
    rows = [44, 0, 17, 17, 3]
    sub64, subbf = oracle.gemm_rows(inputs.bits(A), inputs.bits(B), rows=rows)
    assert np.array_equal(sub64, full64[rows]) and np.array_equal(subbf, fullbf[rows])


def test_bad_row_rejected():
    A, B = inputs.make_problem(4, 4, 8, "normal", seed=1)
    with pytest.raises(ValueError):
        oracle.gemm_rows(inputs.bits(A), inputs.bits(B), rows=[4])


# ---------------------------------------------------------------------------
# Fused epilogue D = alpha * (A B^T) + beta * C + bias
# ---------------------------------------------------------------------------
def test_fused_reduces_to_plain_gemm():
    A, B = inputs.make_problem(23, 41, 57, "normal", seed=13)
    C = inputs.make_operand(23, 41, None, "normal", torch.Generator().manual_seed(14))
    plain64, plainbf = oracle.gemm_rows(inputs.bits(A), inputs.bits(B))
    f64, fbf = oracle.gemm_fused_rows(inputs.bits(A), inputs.bits(B), 1.0, 0.0, C=inputs.bits(C))
    assert np.array_equal(f64, plain64) and np.array_equal(fbf, plainbf)
    f64, fbf = oracle.gemm_fused_rows(inputs.bits(A), inputs.bits(B), 1.0, 0.0)
    assert np.array_equal(fbf, plainbf)


def test_fused_alpha_zero_gives_c_and_bias_exactly():
    g = torch.Generator().manual_seed(15)
    A, B = inputs.make_problem(17, 30, 40, "normal", seed=16)
    C = inputs.make_operand(17, 32, None, "normal", g)          # ldc = 32 > N = 30
    bias = inputs.make_operand(1, 30, None, "uniform", g).reshape(-1)
    _, d = oracle.gemm_fused_rows(inputs.bits(A), inputs.bits(B), 0.0, 1.0, C=inputs.bits(C))
    assert np.array_equal(d, inputs.bits(C)[:, :30])
    _, d = oracle.gemm_fused_rows(inputs.bits(A), inputs.bits(B), 0.0, 0.0, bias=inputs.bits(bias))
    assert np.array_equal(d, np.broadcast_to(inputs.bits(bias), (17, 30)))


def test_fused_bruteforce_tiny_exact():
    rng = np.random.default_rng(200)
    alpha, beta = 0.75, -1.5                                     # exact binary fractions
    for M in (1, 3, 5):
        for N in (1, 2, 6):
            for K in (1, 4, 7):
                A = random_bf16_bits(rng, (M, K))
                B = random_bf16_bits(rng, (N, K))
                C = random_bf16_bits(rng, (M, N + 2))
                bias = random_bf16_bits(rng, (N,))
                ref64, refbf = oracle.gemm_fused_rows(A, B, alpha, beta, C=C, bias=bias, K=K)
                dot = _exact_gemm(A, B, K)
                for m in range(M):
                    for n in range(N):
                        want = (Fraction(alpha) * dot[m][n] + Fraction(beta) * bf16_value(int(C[m, n]))
                                + bf16_value(int(bias[n])))
                        assert Fraction(float(ref64[m, n])) == want, (M, N, K, m, n)
                        assert int(refbf[m, n]) == exact_rne_bf16(want), (M, N, K, m, n)


def test_fused_integer_closed_form():
    A, B = inputs.make_problem(19, 27, 90, "int2", seed=17)
    g = torch.Generator().manual_seed(18)
    C = inputs.make_operand(19, 27, None, "int2", g)
    bias = inputs.make_operand(1, 27, None, "int2", g).reshape(-1)
    ref64, refbf = oracle.gemm_fused_rows(inputs.bits(A), inputs.bits(B), 2.0, -3.0,
                                          C=inputs.bits(C), bias=inputs.bits(bias))
    exact = (2 * (A.to(torch.int64).numpy() @ B.to(torch.int64).numpy().T)
             - 3 * C.to(torch.int64).numpy() + bias.to(torch.int64).numpy()[None, :])
    assert np.array_equal(ref64, exact.astype(np.float64))
    want = np.array([[exact_rne_bf16(Fraction(int(v))) for v in row] for row in exact], dtype=np.uint16)
    assert np.array_equal(refbf, want)
