"""Pins of the CPU oracle against facts fixed outside the oracle itself.

Each test ties one oracle function to something independent of its own code:
values the pages print (tests/golden/), closed forms, brute force, exact
rational arithmetic, or a library routine on a special case.  A plausible slip
(a dropped term, a wrong sign or index, two roundings instead of one, a
transposed operand) makes at least one of them fail.
"""
from fractions import Fraction
import math
import os

import numpy as np
import pytest

import synth
from oracle import oracle as O

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _golden_numbers(name):
    vals = []
    with open(os.path.join(GOLD, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                vals.append(line)
    return vals


def round_fraction_to_f32(fr: Fraction) -> float:
    """Exact rational -> nearest float32 (ties to even), normal range only."""
    if fr == 0:
        return 0.0
    sign = -1.0 if fr < 0 else 1.0
    a = abs(fr)
    e = math.floor(math.log2(a.numerator) - math.log2(a.denominator))
    # fix e so that 2^23 <= a / 2^(e-23) < 2^24
    while a >= Fraction(2) ** (e + 1):
        e += 1
    while a < Fraction(2) ** e:
        e -= 1
    scale = Fraction(2) ** (e - 23)
    m = a / scale
    fl = m.numerator // m.denominator
    rem = m - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    return sign * float(Fraction(fl) * scale)


def round_fraction_to_bits(fr: Fraction, prec: int) -> Fraction:
    """Exact rational -> nearest value with `prec` significant bits (ties to even)."""
    if fr == 0:
        return Fraction(0)
    sign = -1 if fr < 0 else 1
    a = abs(fr)
    e = 0
    while a >= Fraction(2) ** (e + 1):
        e += 1
    while a < Fraction(2) ** e:
        e -= 1
    scale = Fraction(2) ** (e - prec + 1)
    m = a / scale
    fl = m.numerator // m.denominator
    rem = m - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    return sign * Fraction(fl) * scale


# ---------------------------------------------------------------- codebook

def test_codebook_is_the_pages():
    page = [float(v) for v in _golden_numbers("codebook_lloyd_max.txt")]
    assert list(O.CODEBOOK) == page


def test_lloyd_iteration_lands_on_page_centroids():
    """Lloyd's iteration on N(0,1) samples converges to the page's levels (to 0.02).

    The textbook optimum (Max 1960) is +-0.4528, +-1.510; the page rounds 1.510 to 1.52.
    """
    x = np.random.default_rng(0).standard_normal(2_000_000)
    c = O.lloyd_max(x, levels=4, iters=300)
    page = np.array(O.CODEBOOK)
    assert np.all(np.abs(c - page) <= 0.02), c
    assert np.all(np.abs(c - np.array([-1.510, -0.4528, 0.4528, 1.510])) <= 0.01), c
    # distortion of the 4-level Gaussian Lloyd-Max quantizer: 0.1175 (Max 1960)
    assert abs(O.quantizer_mse(x[:400_000], c) - 0.1175) < 0.003
    assert abs(O.quantizer_mse(x[:400_000], page) - 0.1175) < 0.003


def test_lloyd_iteration_on_uniform_gives_uniform_levels():
    """Special case with a closed form: for U(0,1) the optimum levels are (2i+1)/8."""
    x = np.random.default_rng(1).uniform(0, 1, 400_000)
    c = O.lloyd_max(x, levels=4, iters=300, init=[0.1, 0.2, 0.3, 0.4])
    assert np.allclose(c, [0.125, 0.375, 0.625, 0.875], atol=3e-3)


def test_uniform_grid_is_worse_by_the_pages_factor():
    """Page: Lloyd-Max levels cut MSE ~4.2x versus a uniform min-max linear grid.

    With the grid spanning one long row of N(0,1) weights (group 4096) the ratio lands
    near the page's figure; at G = 32 it is much smaller (recorded, not asserted)."""
    x = np.random.default_rng(2).standard_normal(1 << 20)
    ratio = O.uniform_minmax_mse(x, 4096) / O.quantizer_mse(x[:300_000], O.CODEBOOK)
    assert 3.0 < ratio < 6.0, ratio


# ---------------------------------------------------------------- nearest centroid

def test_nearest_centroid_brute_force_and_thresholds():
    z = np.concatenate([np.linspace(-4, 4, 20001), [0.0, -0.0]])
    q = O.nearest_centroid(z)
    C = np.array(O.CODEBOOK)
    for zi, qi in zip(z[::97], q[::97]):
        d = [abs(zi - c) for c in C]
        assert qi == d.index(min(d))                     # brute force, first index on ties
    # thresholds at the midpoints -0.985, 0, 0.985; z = 0 is a tie -> lower index (-0.45)
    assert O.nearest_centroid(np.array([0.0]))[0] == 1
    assert list(O.nearest_centroid(np.array([-3.0, -0.9, -0.1, 0.1, 0.9, 3.0]))) == [0, 1, 1, 2, 2, 3]
    assert list(O.nearest_centroid(np.array([-0.99, -0.98, 0.98, 0.99]))) == [0, 1, 2, 3]


# ---------------------------------------------------------------- OLS

def test_ols_recovers_exact_linear_groups():
    g = np.random.default_rng(3)
    C = np.array(O.CODEBOOK)
    for _ in range(200):
        q = g.integers(0, 4, 32)
        S, Z = g.uniform(0.001, 0.1), g.normal(0, 0.01)
        w = S * C[q] + Z
        if len(set(q)) < 2:
            continue
        S2, Z2 = O.ols_fit(w, C[q])
        assert abs(S2 - S) <= 1e-12 * max(1.0, abs(S)) + 1e-13
        assert abs(Z2 - Z) <= 1e-12


def test_ols_matches_lstsq():
    """Library routine on the same design [C_q, 1]; eps changes S by ~1e-13 relative."""
    g = np.random.default_rng(4)
    C = np.array(O.CODEBOOK)
    for _ in range(100):
        q = g.integers(0, 4, 32)
        w = g.normal(0, 0.02, 32)
        S, Z = O.ols_fit(w, C[q])
        A = np.stack([C[q], np.ones(32)], axis=1)
        (S2, Z2), *_ = np.linalg.lstsq(A, w, rcond=None)
        assert abs(S - S2) <= 1e-9 * abs(S2) + 1e-15
        assert abs(Z - Z2) <= 1e-9 * abs(Z2) + 1e-15


def test_ols_degenerate_group_all_equal_codes():
    """All codes equal: the slope's denominator is eps only -> S = 0, Z = mean(w)."""
    w = np.array([0.01, 0.02, 0.03, 0.04] * 8)
    S, Z = O.ols_fit(w, np.full(32, 0.45))
    assert S == 0.0 and abs(Z - w.mean()) < 1e-15


# ---------------------------------------------------------------- 2-bit quantizer

def _fp16_values(g, lo, hi, n):
    return np.asarray(g.uniform(lo, hi, n), dtype=np.float16).astype(np.float64)


def test_quantizer_reconstructs_groups_built_from_the_codebook():
    """W = S*C[q] + Z with balanced codes and fp16-exact S, Z: codes, S and Z come back."""
    g = np.random.default_rng(5)
    N, K = 8, 256
    C = np.array(O.CODEBOOK)
    q = np.stack([g.permutation(np.repeat(np.arange(4), 8)) for _ in range(N * K // 32)]).reshape(N, K)
    S = _fp16_values(g, 0.005, 0.05, N * K // 32).reshape(N, K // 32)
    Z = _fp16_values(g, -0.01, 0.01, N * K // 32).reshape(N, K // 32)
    W = (np.repeat(S, 32, axis=1) * C[q] + np.repeat(Z, 32, axis=1)).astype(np.float32)
    p = O.quantize_2bit(W, np.zeros(0, np.int32))
    assert np.array_equal(p["q"], q)
    assert np.array_equal(p["scales"], S.astype(np.float16).view(np.uint16))
    assert np.array_equal(p["offsets"], Z.astype(np.float16).view(np.uint16))
    deq = O.dequant_2bit(p)
    assert np.max(np.abs(deq - W)) <= 2 * np.spacing(np.abs(W)).max()


def test_quantizer_group_statistics_by_hand():
    """One group worked by hand: normalise, assign, fit, with numbers computed here directly."""
    w = np.array([0.03, -0.01, 0.0, 0.02] * 8, dtype=np.float32)
    p = O.quantize_2bit(w[None, :], np.zeros(0, np.int32))
    wd = w.astype(np.float64)
    z = (wd - wd.mean()) / wd.std()                      # mean 0.01, std sqrt(0.00025)
    assert np.allclose(z[:4], [1.2649110640673518, -1.2649110640673518, -0.6324555320336759, 0.6324555320336759])
    assert list(p["q"][0, :4]) == [3, 0, 1, 2]
    c = np.array([1.52, -1.52, -0.45, 0.45] * 8)
    S = np.sum((wd - wd.mean()) * (c - c.mean())) / (np.sum((c - c.mean()) ** 2) + 1e-12)
    assert abs(p["S"][0, 0] - S) < 1e-15 and abs(p["Z"][0, 0] - (wd.mean() - S * c.mean())) < 1e-15


def test_quantizer_ignores_anchor_positions():
    """Anchor columns leave their group's fit untouched and store code 0."""
    g = np.random.default_rng(6)
    W = synth.weights(4, 64, 0.02, seed=6)
    anchors = np.array([3, 17, 40], dtype=np.int32)
    p1 = O.quantize_2bit(W, anchors)
    W2 = W.copy()
    W2[:, anchors] = g.normal(0, 5.0, (4, 3)).astype(np.float32)
    p2 = O.quantize_2bit(W2, anchors)
    assert np.array_equal(p1["scales"], p2["scales"]) and np.array_equal(p1["offsets"], p2["offsets"])
    assert np.all(p1["q"][:, anchors] == 0)
    assert np.array_equal(p2["anchor_w"][:, :3], W2[:, anchors].astype(np.float16).view(np.uint16))
    # the dequantized matrix carries the exact fp16 anchor values
    deq = O.dequant_2bit(p2)
    assert np.array_equal(deq[:, anchors], W2[:, anchors].astype(np.float16).astype(np.float32))


def test_all_anchor_group_stores_zero():
    W = synth.weights(2, 64, 0.02, seed=7)
    anchors = np.arange(32, 64, dtype=np.int32)
    p = O.quantize_2bit(W, anchors)
    assert np.all(p["scales"][:, 1] == 0) and np.all(p["offsets"][:, 1] == 0)


# ---------------------------------------------------------------- anchors

def test_anchor_count_floor():
    assert O.anchor_count(256) == 8            # 8.96 -> 8 (floor, not round)
    assert O.anchor_count(4096) == 143
    assert O.anchor_count(11008) == 385
    assert O.anchor_count(8192) == 286
    assert O.anchor_count(28672) == 1003
    assert O.anchor_count(5120) == 179
    assert O.anchor_count(13824) == 483


def test_anchor_selection_finds_outlier_channels():
    K = 512
    W = synth.weights(64, K, 0.02, seed=8)
    out = synth.outlier_channels(K, 0.01, seed=8)
    prof = O.activation_profile(synth.channel_sigma(K, out, 20.0))
    ai = O.select_anchors(W, prof)
    assert len(ai) == O.anchor_count(K) and np.all(np.diff(ai) > 0)
    assert set(out.tolist()) <= set(ai.tolist())


def test_anchor_selection_brute_force_and_ties():
    g = np.random.default_rng(9)
    W = g.normal(0, 1, (5, 200))
    prof = g.uniform(0.5, 2, 200)
    ai = O.select_anchors(W, prof)
    score = [math.sqrt(sum(W[n, c] ** 2 for n in range(5))) * prof[c] for c in range(200)]
    ranked = sorted(range(200), key=lambda c: score[c], reverse=True)[:7]
    assert sorted(ranked) == ai.tolist()
    # equal scores everywhere -> the lowest columns win
    Wt = np.ones((3, 200))
    assert O.select_anchors(Wt, np.ones(200)).tolist() == list(range(7))
    # the score multiplies the column norm by the profile (a weight-only rule picks differently)
    W2 = np.ones((3, 200))
    W2[:, 5] = 3.0
    p2 = np.ones(200)
    p2[[10, 11, 12, 13, 14, 15, 16]] = 4.0
    assert O.select_anchors(W2, p2).tolist() == [10, 11, 12, 13, 14, 15, 16]


def test_activation_profile_is_mean_abs_of_gaussian_channels():
    """mean|X_c| of zero-mean Gaussian samples with std sigma_c, against the analytic profile.

    The profile enters the otf-llm README's impact score (section 4) as mean|X_c|.  Samples
    drawn with known sigma give the mean absolute value directly; the analytic form must sit
    within three standard errors of it for every sigma.  sqrt(pi/2)*sigma, sigma**2 or a
    missing square root each land hundreds of standard errors away.
    """
    g = np.random.default_rng(31)
    sig = np.array([0.25, 1.0, 3.0, 20.0])
    n = 400_000
    X = g.normal(0.0, 1.0, (n, len(sig))) * sig
    mean_abs = np.mean(np.abs(X), axis=0)
    se = np.std(np.abs(X), axis=0, ddof=1) / math.sqrt(n)
    prof = O.activation_profile(sig)
    assert np.all(np.abs(prof - mean_abs) <= 3.0 * se), (prof, mean_abs, se)


def test_anchor_selection_with_unequal_channel_sigmas_matches_sampled_profile():
    """Columns whose norms and activation sigmas both vary: the oracle's choice from the
    analytic profile equals a brute-force choice from sampled mean|X_c|.

    The test matrix is built so that scoring with sigma_c**2 (or a norm-only rule) picks a
    different set: column norms fall as sigma rises, so the product decides the ranking.
    """
    g = np.random.default_rng(32)
    K, N = 200, 16
    sigma = np.linspace(0.5, 6.0, K)
    g.shuffle(sigma)
    W = g.normal(0.0, 1.0, (N, K))
    W /= np.sqrt(np.sum(W * W, axis=0))                  # unit column norms
    W *= (30.0 / sigma) ** 0.5 * (1.0 + 0.4 * g.uniform(size=K))   # norms fall as sigma rises
    A = O.anchor_count(K)
    n = 200_000
    X = g.normal(0.0, 1.0, (n, K)) * sigma
    sampled = np.mean(np.abs(X), axis=0)
    score = [math.sqrt(sum(float(W[r, c]) ** 2 for r in range(N))) * float(sampled[c]) for c in range(K)]
    brute = sorted(sorted(range(K), key=lambda c: (-score[c], c))[:A])
    got = O.select_anchors(W, O.activation_profile(sigma)).tolist()
    assert got == brute
    # the same matrix scored with sigma squared or with the norm alone picks other columns
    assert O.select_anchors(W, sigma ** 2).tolist() != got
    assert O.select_anchors(W, np.ones(K)).tolist() != got


# ---------------------------------------------------------------- packing

def test_pack_2bit_worked_examples():
    for line in _golden_numbers("pack_2bit_worked.txt"):
        lhs, rhs = line.split("->")
        q = np.array([[int(v) for v in lhs.split()]], dtype=np.uint8)
        assert O.pack_2bit(q)[0, 0] == int(rhs.strip(), 16)


def test_pack_roundtrip_and_sizes():
    g = np.random.default_rng(10)
    q = g.integers(0, 4, (7, 256)).astype(np.uint8)
    b = O.pack_2bit(q)
    assert b.shape == (7, 64) and np.array_equal(O.unpack_2bit(b), q)
    q4 = g.integers(0, 16, (7, 256)).astype(np.uint8)
    b4 = O.pack_nf4(q4)
    assert b4.shape == (7, 128) and np.array_equal(O.unpack_nf4(b4), q4)
    assert O.pack_nf4(np.array([[1, 2]], np.uint8))[0, 0] == 0x21


def test_bits_per_weight():
    """2 bits of code + 2 fp16 per group of 32 = 3.0 bits; anchors add 16*A/K bits."""
    def bits(N, K):
        A = O.anchor_count(K)
        byts = N * K / 4 + 2 * 2 * N * K / 32 + 2 * N * A + 4 * A
        return 8 * byts / (N * K)
    assert abs(bits(512, 256) - 3.5) < 0.01
    assert abs(bits(4096, 4096) - 3.56) < 0.01
    assert abs(bits(4096, 11008) - 3.56) < 0.01
    # NF4: 4 bits + fp32 per 64 -> 4.5 bits = 28.125% of fp16 (codes alone: 25%)
    assert (4 + 32 / 64) / 16 == 0.28125


# ---------------------------------------------------------------- NF4

def test_nf4_table_matches_construction_and_publication():
    T = O.nf4_table()
    pub = np.array([float(v) for v in _golden_numbers("nf4_levels_qlora.txt")], dtype=np.float32)
    assert np.array_equal(T.view(np.uint32), pub.view(np.uint32))
    cons = O.nf4_table_construction()
    assert np.max(np.abs(cons - T.astype(np.float64))) < 1e-6
    assert T[0] == -1.0 and T[15] == 1.0 and T[7] == 0.0
    assert np.all(np.diff(T) > 0)
    assert np.sum(T < 0) == 7 and np.sum(T > 0) == 8


def test_nf4_quantizer_recovers_table_points_and_zero_block():
    g = np.random.default_rng(11)
    T = O.nf4_table().astype(np.float64)
    q = g.integers(0, 16, (4, 128))
    q[:, 0] = 15                                         # each block's max is +absmax
    q[:, 64] = 0
    am = g.uniform(0.01, 0.1, (4, 2))
    W = (T[q] * np.repeat(am, 64, axis=1)).astype(np.float32)
    p = O.quantize_nf4(W)
    assert np.array_equal(p["q"], q)
    assert np.array_equal(p["absmax"], np.max(np.abs(W.reshape(4, 2, 64)), axis=2))
    Wz = np.zeros((1, 64), np.float32)
    pz = O.quantize_nf4(Wz)
    assert np.all(pz["q"] == 7) and np.all(O.dequant_nf4(pz) == 0)


def test_nf4_nearest_level_brute_force():
    W = synth.weights(3, 128, 0.02, seed=12)
    p = O.quantize_nf4(W)
    T = O.nf4_table().astype(np.float64)
    for n in range(3):
        for k in range(0, 128, 5):
            am = float(p["absmax"][n, k // 64])
            r = float(W[n, k]) / am
            d = [abs(r - t) for t in T]
            assert p["q"][n, k] == d.index(min(d))


# ---------------------------------------------------------------- dequant rounding

def test_dequant_2bit_is_one_fused_rounding():
    """fmaf(S, C[q], Z) equals the exactly rounded S*C[q]+Z; two roundings would differ."""
    g = np.random.default_rng(13)
    C32 = [Fraction(float(np.float32(c))) for c in O.CODEBOOK]
    L = O._lib()
    mism_two = 0
    for _ in range(4000):
        s = np.float16(g.uniform(-0.1, 0.1))
        z = np.float16(g.uniform(-0.05, 0.05))
        q = int(g.integers(0, 4))
        got = L.oracle_dequant_2bit_one(int(s.view(np.uint16)), q, int(z.view(np.uint16)))
        exact = Fraction(float(s)) * C32[q] + Fraction(float(z))
        assert got == round_fraction_to_f32(exact) if exact != 0 else got == 0.0
        two = np.float32(np.float32(np.float32(s) * np.float32(O.CODEBOOK[q])) + np.float32(z))
        mism_two += (two != np.float32(got))
    assert mism_two > 0          # the test data does separate one rounding from two


def test_dequant_matrix_layout():
    """Column k of row n reads byte k/4 bits 2(k%4); group k/32; by hand on a small matrix."""
    g = np.random.default_rng(14)
    N, K = 3, 64
    q = g.integers(0, 4, (N, K)).astype(np.uint8)
    sc = np.asarray(g.uniform(0.01, 0.05, (N, 2)), np.float16)
    of = np.asarray(g.uniform(-0.01, 0.01, (N, 2)), np.float16)
    p = dict(codes=O.pack_2bit(q), scales=sc.view(np.uint16), offsets=of.view(np.uint16),
             anchor_idx=np.array([5], np.int32), anchor_w=np.full((N, 8), np.float16(0.25).view(np.uint16), np.uint16),
             A=1, ld_anchor=8, N=N, K=K)
    d = O.dequant_2bit(p)
    for n in range(N):
        for k in range(K):
            if k == 5:
                assert d[n, k] == 0.25
                continue
            exact = Fraction(float(sc[n, k // 32])) * Fraction(float(np.float32(O.CODEBOOK[q[n, k]]))) + Fraction(float(of[n, k // 32]))
            assert d[n, k] == round_fraction_to_f32(exact)


def test_dequant_nf4_one_rounding():
    g = np.random.default_rng(15)
    N, K = 2, 128
    q = g.integers(0, 16, (N, K)).astype(np.uint8)
    am = g.uniform(0.01, 0.2, (N, 2)).astype(np.float32)
    p = dict(codes=O.pack_nf4(q), absmax=am, N=N, K=K)
    d = O.dequant_nf4(p)
    T = O.nf4_table()
    for n in range(N):
        for k in range(0, K, 3):
            exact = Fraction(float(T[q[n, k]])) * Fraction(float(am[n, k // 64]))
            assert d[n, k] == (round_fraction_to_f32(exact) if exact != 0 else 0.0)


def test_output_rounding_matches_ieee_rne():
    g = np.random.default_rng(16)
    v = np.concatenate([g.normal(0, 1, 20000), g.normal(0, 1e-5, 2000), g.normal(0, 3e4, 2000),
                        [65504, 65519.99, 65520, 1 + 2 ** -11, 1 + 3 * 2 ** -11, 2 ** -25, 2 ** -24 * 1.5, 0.0]]).astype(np.float32)
    h = O.round_to(v, "f16")
    assert np.array_equal(h, v.astype(np.float16).view(np.uint16))          # library RNE
    b = O.round_to(v, "bf16")
    for x, bits in zip(v[::37], b[::37]):
        ref = round_fraction_to_bits(Fraction(float(x)), 8)
        got = np.array([int(bits) << 16], dtype=np.uint32).view(np.float32)[0]
        assert float(got) == float(ref)


# ---------------------------------------------------------------- matmul

def test_matmul_ref_against_exact_sums():
    g = np.random.default_rng(17)
    for (M, N, K) in [(1, 4, 32), (3, 5, 96), (2, 16, 256)]:
        W = g.normal(0, 0.02, (N, K)).astype(np.float32)
        x = synth.activations(M, K, "f16", seed=int(K))
        y, E = O.matmul_ref(W, x, "f16")
        xv = O.x_values(x, "f16")
        for m in range(M):
            for n in range(N):
                prods = [Fraction(float(W[n, k])) * Fraction(float(xv[m, k])) for k in range(K)]
                exact = sum(prods)
                assert abs(y[m, n] - float(exact)) <= 1e-12 * E[m, n]
                assert abs(E[m, n] - math.fsum(abs(float(p)) for p in prods)) <= 1e-12 * E[m, n]


def test_matmul_ref_is_not_transposed():
    W = np.zeros((2, 32), np.float32)
    W[1, 3] = 1.0
    x = np.zeros((1, 32), np.float16)
    x[0, 3] = 2.0
    y, _ = O.matmul_ref(W, x.view(np.uint16), "f16")
    assert y.tolist() == [[0.0, 2.0]]


def test_row_error_scale_equals_matmul_error_scale():
    """The sampled parity tests take their tolerance scale from row_error_scale (numpy);
    it must equal the compiled matmul_ref's E for both x dtypes, and equal |y| when every
    product is non-negative (E is then the sum itself)."""
    g = np.random.default_rng(33)
    for (M, N, K) in [(1, 3, 64), (4, 7, 256), (2, 5, 512)]:
        W = g.normal(0, 0.02, (N, K)).astype(np.float32)
        for xdt in ("f16", "bf16"):
            x = synth.activations(M, K, xdt, seed=K + M)
            _, E = O.matmul_ref(W, x, xdt)
            Er = O.row_error_scale(W, x, xdt)
            assert Er.shape == E.shape
            assert np.all(np.abs(Er - E) <= 1e-12 * E)
    Wp = np.abs(g.normal(0, 1, (3, 96))).astype(np.float32)
    xp = np.abs(g.normal(0, 1, (2, 96))).astype(np.float16).view(np.uint16)
    y, _ = O.matmul_ref(Wp, xp, "f16")
    assert np.all(np.abs(O.row_error_scale(Wp, xp, "f16") - y) <= 1e-12 * y)
    # flipping the sign of W or x leaves E unchanged
    assert np.array_equal(O.row_error_scale(-Wp, xp, "f16"), O.row_error_scale(Wp, xp, "f16"))


def test_row_gemv_matches_full_matmul():
    W = synth.weights(40, 256, 0.02, seed=18)
    ai = O.select_anchors(W, np.ones(256))
    p = O.quantize_2bit(W, ai)
    x = synth.activations(3, 256, "bf16", seed=18)
    y, _ = O.matmul_ref(O.dequant_2bit(p), x, "bf16")
    assert np.array_equal(O.gemv_2bit_rows(p, x, "bf16", 10, 30), y[:, 10:30])
    pn = O.quantize_nf4(W)
    yn, _ = O.matmul_ref(O.dequant_nf4(pn), x, "bf16")
    assert np.array_equal(O.gemv_nf4_rows(pn, x, "bf16", 0, 40), yn)


def test_page_decode_ceilings():
    """The README's ceilings are bus bandwidth divided by bytes per token."""
    for line in _golden_numbers("page_roofline.txt"):
        bw, gb, claim, rel = line.split()
        tps = float(bw) / float(gb)
        if rel == "approx":
            assert abs(tps - float(claim)) / float(claim) < 0.05
        else:
            assert tps >= float(claim)


# ---------------------------------------------------------------- v3.2 INT4 (uniform grid, permutation, 1% outliers)

def test_int4_grid_points_recovered_exactly():
    """Groups built as S16 * q with q on the symmetric grid (each group holding a +-7, so
    its max |w| is 7 * S16) come back with the same codes and the same binary16 scale."""
    g = np.random.default_rng(40)
    N, K = 6, 256
    S16 = g.uniform(0.001, 0.05, (N, K // 32)).astype(np.float16)
    q = g.integers(-7, 8, (N, K)).astype(np.int8)
    q[:, ::32] = np.where(g.random((N, K // 32)) < 0.5, -7, 7)
    W = (S16.astype(np.float32).repeat(32, axis=1) * q.astype(np.float32)).astype(np.float32)
    p = O.quantize_int4(W, np.arange(K, dtype=np.int32), np.zeros(0, np.int32))
    assert np.array_equal(p["q"], q)
    assert np.array_equal(p["scales"], S16.view(np.uint16))
    assert np.array_equal(O.dequant_int4(p), W)


def test_int4_pack_roundtrip_and_worked_byte():
    g = np.random.default_rng(41)
    q = g.integers(-8, 8, (5, 64)).astype(np.int8)
    b = O.pack_int4(q)
    assert b.shape == (5, 32) and np.array_equal(O.unpack_int4(b), q)
    # position 0 = -1 (two's complement 0xF) in the low nibble, position 1 = 3 in the high nibble
    assert O.pack_int4(np.array([[-1, 3]], np.int8))[0, 0] == 0x3F
    assert O.pack_int4(np.array([[7, -8]], np.int8))[0, 0] == 0x87


def test_int4_permutation_orders_by_score_and_inverts():
    g = np.random.default_rng(42)
    N, K = 9, 160
    W = g.normal(0, 1, (N, K))
    prof = g.uniform(0.5, 3.0, K)
    perm = O.int4_permutation(W, prof)
    assert sorted(perm.tolist()) == list(range(K))                     # a permutation
    score = [math.sqrt(sum(W[n, c] ** 2 for n in range(N))) * prof[c] for c in range(K)]
    assert all(score[perm[j]] >= score[perm[j + 1]] for j in range(K - 1))
    inv = np.empty(K, np.int64)
    inv[perm] = np.arange(K)
    x = g.normal(0, 1, K)
    assert np.array_equal(x[perm][inv], x)                              # the inverse undoes it
    assert abs(W[:, perm] @ x[perm] - W @ x).max() < 1e-12 * np.abs(W).sum()   # y is unchanged
    # equal scores keep the columns in order
    assert O.int4_permutation(np.ones((2, 40)), np.ones(40)).tolist() == list(range(40))


def test_int4_dequant_places_values_at_permuted_columns_and_keeps_zero():
    """W_eff[n][perm[j]] = S * q[n][j]; anchors store q = 0 and are replaced by their binary16
    value; a zero weight reconstructs to exactly 0 (zero-point 0)."""
    K = 64
    perm = np.r_[np.arange(32, 64), np.arange(0, 32)].astype(np.int32)
    W = np.zeros((2, K), np.float32)
    W[0, 40] = 0.7                     # permuted position 8, group 0
    W[0, 3] = -0.35                    # permuted position 35, group 1
    W[1, 33] = 5.0                     # anchor column
    W[1, 10] = 0.02
    anchors = np.array([33], np.int32)
    p = O.quantize_int4(W, perm, anchors)
    assert p["q"][1, 1] == 0           # column 33 sits at permuted position 1
    Wd = O.dequant_int4(p)
    assert Wd[1, 33] == np.float32(np.float16(5.0))
    assert Wd[0, 40] == np.float32(np.float16(0.1)) * 7 and p["q"][0, 8] == 7
    assert Wd[0, 3] == np.float32(np.float16(0.05)) * -7
    zero_cols = [c for c in range(K) if W[0, c] == 0 and c not in (33,)]
    assert np.all(Wd[0, zero_cols] == 0.0)


def test_int4_rounding_error_bound():
    """Every non-anchor weight lands within half a grid step of its reconstruction, or is
    clipped at +-7 steps (only when the binary16 scale rounded below max|w|/7)."""
    W = synth.weights(48, 512, 0.02, seed=43, big_frac=0.002, big_mult=10.0)
    prof = np.ones(512)
    perm = O.int4_permutation(W, prof)
    ai = O.select_anchors(W, prof, frac=O.INT4_OUTLIER_FRAC)
    p = O.quantize_int4(W, perm, ai)
    Wd = O.dequant_int4(p).astype(np.float64)
    S = p["scales"].view(np.float16).astype(np.float64).repeat(32, axis=1)[:, np.argsort(perm)]
    err = np.abs(W.astype(np.float64) - Wd)
    allow = np.maximum(S / 2, np.abs(W) - 7 * S) * (1 + 1e-12)
    nonanchor = np.ones(512, bool)
    nonanchor[ai] = False
    assert np.all(err[:, nonanchor] <= allow[:, nonanchor])
    assert np.all(Wd[:, ai] == W[:, ai].astype(np.float16).astype(np.float64))


def test_int4_outlier_count_and_bits_per_weight():
    """Top-1% outlier columns (floor), and 4 bits + one binary16 scale per 32 = 4.5 bits per
    weight before the outliers (1% binary16 columns add 0.16 bit at these sizes)."""
    for K, A in [(256, 2), (4096, 40), (11008, 110), (8192, 81), (28672, 286)]:
        assert int(np.floor(O.INT4_OUTLIER_FRAC * K)) == A
    N, K = 4096, 4096
    A = int(np.floor(O.INT4_OUTLIER_FRAC * K))
    bits = 8 * (N * K / 2 + 2 * N * K / 32 + 2 * N * A + 4 * A + 4 * K) / (N * K)
    assert abs((4 + 16 / 32) - 4.5) < 1e-12 and abs(bits - 4.66) < 0.01


# ---------------------------------------------------------------- NF4 double quantization (QLoRA)

def _rn_f32(r: Fraction) -> np.float32:
    """Exact rational -> nearest fp32 (ties to even), checked against both fp32 neighbours."""
    f = np.float32(float(r))
    cands = [np.nextafter(f, np.float32(-np.inf)), f, np.nextafter(f, np.float32(np.inf))]
    best = min(cands, key=lambda c: (abs(Fraction(float(c)) - r), int(np.float32(c).view(np.uint32)) & 1))
    return np.float32(best)


def test_e4m3_decode_matches_the_library_and_the_format_definition():
    torch = pytest.importorskip("torch")
    lib = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    ours = O.e4m3_decode(np.arange(256, dtype=np.uint8))
    assert np.array_equal(np.isnan(ours), np.isnan(lib)) and np.isnan(ours).sum() == 2
    ok = ~np.isnan(ours)
    assert np.array_equal(ours[ok], lib[ok])
    # the format's landmarks: largest finite, smallest normal, smallest subnormal, one, sign
    assert ours[0x7E] == 448.0 and ours[0x08] == 2.0 ** -6 and ours[0x01] == 2.0 ** -9
    assert ours[0x38] == 1.0 and ours[0xC0] == -2.0 and ours[0x80] == 0.0


def test_e4m3_encode_is_the_nearest_code_with_ties_to_even():
    torch = pytest.importorskip("torch")
    g = np.random.default_rng(7)
    vals = np.concatenate([g.standard_normal(3000) * 10.0 ** g.uniform(-4, 2.5, 3000),
                           (O.e4m3_decode(np.arange(1, 0x7E)) + O.e4m3_decode(np.arange(2, 0x7F))) / 2,  # midpoints
                           [0.0, 2.0 ** -10, 3 * 2.0 ** -10, 463.99, -463.99]])
    vals = vals[np.abs(vals) < 464.0]
    ours = O.e4m3_encode(vals)
    lib = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    # (+-0: the library keeps the sign of a value that rounds to zero; compare magnitudes there)
    zero = O.e4m3_decode(ours) == 0
    assert np.array_equal(ours[~zero], lib[~zero]) and np.all(lib[zero] & 0x7F == 0)
    # beyond the largest finite value the reading saturates (the library gives NaN there)
    assert O.e4m3_encode(np.array([448.0, 464.0, 1e6, -1e6])).tolist() == [0x7E, 0x7E, 0x7E, 0xFE]


def test_nf4_double_quant_blocks_mean_and_error_bound():
    """Second-level blocks are 256 consecutive maxima in row-major order; each element is
    reconstructed within half an E4M3 step of (c - mean) / s2, times s2, plus fp32 rounding."""
    N, KB = 96, 8                                   # 768 first-level maxima -> 3 blocks
    g = np.random.default_rng(3)
    c = (0.01 + 0.05 * g.random((N, KB))).astype(np.float32)
    c[32:64] *= 4                                   # rows 32..63 are block 1 (256 = 32 rows x 8)
    acodes, second = O.double_quantize_absmax(c)
    mean = np.float32(np.sum(c.astype(np.float64)) / c.size)
    assert second[0] == mean and len(second) == 1 + 3
    flat = c.ravel().astype(np.float64)
    for j in range(3):
        seg = flat[256 * j:256 * (j + 1)] - np.float64(mean)
        assert second[1 + j] == np.float32(np.max(np.abs(seg)) / 448.0)
    assert second[2] > 2 * max(second[1], second[3])
    v = (flat - np.float64(mean)) / np.repeat(second[1:].astype(np.float64), 256)
    dec = O.e4m3_decode(acodes.ravel())
    half_step = np.where(np.abs(v) >= 2.0 ** -6, 2.0 ** (np.floor(np.log2(np.maximum(np.abs(v), 2.0 ** -6))) - 4), 2.0 ** -10)
    assert np.all(np.abs(dec - v) <= half_step * (1 + 1e-12))
    # the block maximum maps to +-448 exactly
    for j in range(3):
        i = 256 * j + int(np.argmax(np.abs(v[256 * j:256 * (j + 1)])))
        assert abs(dec[i]) == 448.0


def test_nf4_double_quant_dequant_is_two_exact_roundings():
    """W = RN32(T[q] * RN32(E4M3(acode) * s2 + mean)) on every element of a small case,
    the roundings done here on exact rationals."""
    W = synth.weights(6, 128, 0.02, seed=11, big_frac=0.01, big_mult=10.0)
    p = O.quantize_nf4_dq(W)
    got = O.dequant_nf4_dq(p)
    T = O.nf4_table()
    q = O.unpack_nf4(p["codes"])
    dec = O.e4m3_decode(p["acodes"])
    mean, s2 = p["second"][0], p["second"][1:]
    for n in range(6):
        for k in range(128):
            i = n * 2 + k // 64
            cp = _rn_f32(Fraction(float(dec[n, k // 64])) * Fraction(float(s2[i // 256])) + Fraction(float(mean)))
            w = _rn_f32(Fraction(float(T[q[n, k]])) * Fraction(float(cp)))
            assert got[n, k] == w, (n, k)


def test_nf4_double_quant_degenerate_blocks_and_bits_per_weight():
    # every maximum equal to the mean: s2 = 0, codes 0, reconstruction = the mean exactly
    c = np.full((4, 64), 0.037, dtype=np.float32)
    acodes, second = O.double_quantize_absmax(c)
    assert np.all(acodes == 0) and np.all(second[1:] == 0)
    p = dict(codes=np.zeros((4, 2048), np.uint8) + 0x77, acodes=acodes, second=second, N=4, K=4096)
    assert np.all(O.dequant_nf4_dq(p) == np.float32(O.nf4_table()[7]) * np.float32(0.037))
    # storage: 4 bits + 8 bits per 64 + 32 bits per 64*256 (+ one mean) = 4.127 bits per weight
    N, K = 4096, 4096
    bits = 8 * (N * K / 2 + N * K / 64 + 4 * (N * K / 64 / 256 + 1)) / (N * K)
    assert abs(bits - (4 + 8 / 64 + 32 / (64 * 256))) < 1e-5 and abs(bits - 4.127) < 1e-3
