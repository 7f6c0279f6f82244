"""CPU checks of the readings the GPU quantizers rest on (no GPU):

* the summation orders of numpy's reductions, which the oracle's quantizers use and the
  GPU kernels reproduce operation for operation: along a row, pairwise with eight
  interleaved partial sums; down a column, row by row;
* the NF4 nearest level from the two levels around r only;
* the 2-bit nearest level from the side of the level midpoints that d * (1/sd) falls on,
  with the exact quotient near a midpoint.
Each restated decision is compared with the oracle's full argmin on values dense around
every decision point (a few ulps either side), where a shortcut would go wrong first."""
import numpy as np

from oracle import oracle as O


def pairwise8(a):
    n = len(a)
    if n < 8:
        r = 0.0
        for v in a:
            r += v
        return r
    r = list(a[:8])
    i = 8
    while i < n - n % 8:
        for j in range(8):
            r[j] += a[i + j]
        i += 8
    res = ((r[0] + r[1]) + (r[2] + r[3])) + ((r[4] + r[5]) + (r[6] + r[7]))
    while i < n:
        res += a[i]
        i += 1
    return 0.0 + res


def test_numpy_row_sums_are_pairwise_by_eight():
    rng = np.random.default_rng(0)
    for n in range(1, 33):
        A = rng.standard_normal((300, n)) * np.exp(3 * rng.standard_normal((300, n)))
        ref = A.sum(axis=1)
        for i in range(300):
            assert pairwise8(list(A[i])) == ref[i], (n, i)
        assert np.array_equal(A.mean(axis=1), np.array([pairwise8(list(r)) / n for r in A]))


def test_numpy_column_sums_are_row_by_row():
    rng = np.random.default_rng(1)
    for N, K in [(3000, 40), (9, 700)]:
        W = rng.standard_normal((N, K)) * np.exp(2 * rng.standard_normal((N, K)))
        acc = np.zeros(K)
        for n in range(N):
            acc = acc + W[n] * W[n]
        assert np.array_equal(acc, np.sum(W * W, axis=0))


def _around(points, ulps=6):
    out = []
    for p in points:
        v = np.float64(p)
        for _ in range(ulps):
            v = np.nextafter(v, -np.inf)
        for _ in range(2 * ulps + 1):
            out.append(v)
            v = np.nextafter(v, np.inf)
    return np.array(out)


def test_nf4_two_level_bracket_equals_full_argmin():
    T = O.nf4_table().astype(np.float64)
    mids = (T[:-1] + T[1:]) / 2
    r = np.concatenate([_around(mids), _around(T), np.linspace(-1, 1, 20001)])
    r = r[(r >= -1) & (r <= 1)]
    full = np.argmin(np.abs(r[:, None] - T), axis=1)
    for x, q in zip(r, full):
        i = 0
        for step in (8, 4, 2, 1):
            if T[i + step] <= x:
                i += step
        if i < 15:
            d0, d1 = abs(x - T[i]), abs(x - T[i + 1])
            i = i + 1 if d1 < d0 else i
        assert i == q, (x, i, q)


def test_2bit_midpoint_side_equals_exact_decision():
    """The kernel's decision: z' = d * fl(1/sd); outside 1e-9 of the midpoints -0.985, 0, 0.985 the side
    of z' decides, otherwise d / sd and the four distances do.  Compared with the oracle on the
    exact quotient, for d/sd dense around every midpoint and spread over the range."""
    rng = np.random.default_rng(2)
    C = np.asarray(O.CODEBOOK, dtype=np.float64)
    for sd in [0.0137, 1.0, 3.3e-5, 7.77, float(rng.uniform(1e-3, 1e-1))]:
        inv = 1.0 / sd
        targets = np.concatenate([_around([-0.985, 0.0, 0.985], ulps=40), rng.uniform(-6, 6, 4000)])
        for t in targets:
            d = t * sd                                   # a numerator whose quotient lands near t
            z = d / sd
            exact = int(O.nearest_centroid(np.array([z]))[0])
            za = d * inv
            mag = abs(za)
            if mag > 1e-9 and (mag < 0.985 - 1e-9 or mag > 0.985 + 1e-9):
                outer = 1 if mag > 0.985 else 0
                got = (1 - outer) if za < 0 else (2 + outer)
            else:
                got = int(np.argmin(np.abs(z - C)))
            assert got == exact, (sd, t, got, exact)
