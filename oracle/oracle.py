"""CPU oracle for the low-bit linear layer — TEST INFRASTRUCTURE, not the product.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg
may import this module.  The GPU library never calls it, and it shares no code
with the GPU library: its dequantization and products live in ``lq_oracle.c``,
its quantizers below, all written from the definitions on the pages.

Functions and what they follow
------------------------------
* ``CODEBOOK``, ``lloyd_max``        otf-llm 4.0.1 README, section 2, "The Lloyd-Max
                                      Non-Uniform Solution" (MSQE objective, 4 levels).
* ``uniform_minmax_mse``             same section, "Why Uniform Linear 2-Bit
                                      Quantization Fails" (the min-max linear grid).
* ``nearest_centroid``               section 3 "assigned centroids C_q"; assignment is
                                      nearest centroid after per-group mean/std
                                      normalisation (the pages leave the rule open).
* ``ols_fit``                        section 3, "Closed-Form Group Linear Regression
                                      (S_g, Z_g)", the two closed-form equations.
* ``select_anchors``                 section 4, "Profile-Guided Activation Outliers":
                                      impact score I_c = ||W[:,c]||_2 * mean|X_c|, top 3.5%.
* ``quantize_2bit``                  sections 3 and 4 together, groups of G = 32 along K.
* ``pack_2bit`` / ``unpack_2bit``    "Key v4.0 Innovations": 4 two-bit codes per uint8.
* ``nf4_table`` / ``quantize_nf4``   AirQuant README, "Fundamentacao Teorica" item 2
                                      (NF4, block-wise) and its QLoRA reference.
* ``pack_nf4`` / ``unpack_nf4``      NF4 storage, 2 codes per byte.
* ``dequant_2bit`` / ``dequant_nf4`` the reconstruction S*C[q]+Z / T[q]*absmax (C code).
* ``int4_permutation``, ``quantize_int4``, ``pack_int4`` / ``unpack_int4``, ``dequant_int4``
                                     the otf-llm README's v3.2 INT4 engine ("Comparative
                                      Analysis: INT4 (v3.2) vs INT2 Non-Uniform (v4.0)" and
                                      the "Method Comparison Table"): 2 weights per byte,
                                      uniform grid, zero-point 0, a global static column
                                      permutation, top-1% FP16 outlier columns.
* ``e4m3_decode`` / ``e4m3_encode``, ``double_quantize_absmax``, ``quantize_nf4_dq``,
  ``dequant_nf4_dq``                 NF4 double quantization, from the QLoRA method the
                                      AirQuant README cites for NF4: the fp32 block maxima
                                      quantized again as 8-bit floats (E4M3) in blocks of
                                      256, after subtracting their mean.
* ``matmul_ref``                     y = x * W_eff^T in fp64, with the error scale
                                      E = |x| * |W_eff|^T.

Parity: every function above is pinned by ``tests/test_oracle_pins.py`` against
facts the pages or mathematics fix (published constants, closed forms, brute force,
exact rational arithmetic, library routines on special cases).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from pathlib import Path

import numpy as np

_HERE = Path(__file__).resolve().parent

# ---------------------------------------------------------------------------
# Constants the pages fix
# ---------------------------------------------------------------------------

#: otf-llm README, section 2: the four Lloyd-Max centroids, in listed order.
CODEBOOK = (-1.52, -0.45, 0.45, 1.52)
#: Group size along K (otf-llm README section 3, "small blocks (G=32)").
GROUP = 32
#: Anchor fraction (otf-llm README section 4 "Top-3.5%", and the converter's CLI argument 0.035).
ANCHOR_FRAC = 0.035
#: NF4 block size along K.
NF4_BLOCK = 64
#: OLS denominator epsilon (the page writes "+ eps" without a value).
OLS_EPS = 1e-12
#: v3.2 INT4 engine: outlier fraction ("Top-1% FP16 Outlier Channels"), group size along the
#: permuted columns and the symmetric grid's largest code (readings; the page gives only
#: "2 weights / byte", "Uniform Linear Grid" and "Symmetric Zero-Point = 0").
INT4_OUTLIER_FRAC = 0.01
INT4_GROUP = 32
INT4_QMAX = 7

#: The NF4 levels as published with the QLoRA data type (Dettmers et al. 2023,
#: the paper the AirQuant README cites for NF4), as float32.  ``nf4_table_construction``
#: rebuilds them from their definition and the pin test checks the two agree.
_NF4_PUBLISHED = (
    -1.0, -0.6961928009986877, -0.5250730514526367, -0.39491748809814453,
    -0.28444138169288635, -0.18477343022823334, -0.09105003625154495, 0.0,
    0.07958029955625534, 0.16093020141124725, 0.24611230194568634, 0.33791524171829224,
    0.44070982933044434, 0.5626170039176941, 0.7229568362236023, 1.0,
)


def nf4_table() -> np.ndarray:
    """The 16 NF4 levels (float32, ascending)."""
    return np.array(_NF4_PUBLISHED, dtype=np.float32)


def nf4_table_construction() -> np.ndarray:
    """NF4 levels from their definition, in float64.

    The data type places levels at quantiles of N(0,1): 8 on the positive side and
    7 on the negative side, at evenly spaced probabilities between 1/2 and an
    outer probability p_out, plus an exact zero, all divided by the largest so the
    range is [-1, 1].  p_out sits halfway between the outer quantile points of a
    15- and a 16-level symmetric grid: p_out = 1 - (1/(2*15) + 1/(2*16)) / 2.
    """
    from scipy.stats import norm
    p_out = 1.0 - 0.5 * (1.0 / 30.0 + 1.0 / 32.0)
    pos = norm.ppf(np.linspace(p_out, 0.5, 9)[:-1])    # 8 positive quantiles
    neg = -norm.ppf(np.linspace(p_out, 0.5, 8)[:-1])   # 7 negative quantiles
    levels = np.sort(np.concatenate([neg, [0.0], pos]))
    return levels / np.max(levels)


# ---------------------------------------------------------------------------
# The compiled part (dequantization and fp64 products)
# ---------------------------------------------------------------------------

_LIB = None


def lib_path() -> Path:
    return _HERE / "_build" / "liblq_oracle.so"


def build(force: bool = False) -> Path:
    """Compile lq_oracle.c with gcc (no vector intrinsics, no contraction)."""
    out = lib_path()
    src = _HERE / "lq_oracle.c"
    if out.exists() and not force and out.stat().st_mtime >= src.stat().st_mtime:
        return out
    out.parent.mkdir(parents=True, exist_ok=True)
    tmp = out.with_suffix(f".{os.getpid()}.tmp")
    subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
                    "-fvisibility=hidden", str(src), "-o", str(tmp), "-lm"], check=True)
    os.replace(tmp, out)
    return out


def _lib():
    global _LIB
    if _LIB is None:
        path = build()
        L = ctypes.CDLL(str(path))
        P = ctypes.c_void_p
        i = ctypes.c_int
        L.oracle_dequant_2bit.argtypes = [P, P, P, P, P, i, i, i, i, P]
        L.oracle_dequant_nf4.argtypes = [P, P, P, i, i, P]
        L.oracle_dequant_int4.argtypes = [P, P, P, P, P, i, i, i, i, P]
        L.oracle_dequant_nf4_dq.argtypes = [P, P, P, P, i, i, P]
        L.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
        L.oracle_e4m3_to_double.restype = ctypes.c_double
        L.oracle_double_to_e4m3.argtypes = [ctypes.c_double]
        L.oracle_double_to_e4m3.restype = ctypes.c_uint8
        L.oracle_round_f32.argtypes = [P, ctypes.c_size_t, i, P]
        L.oracle_matmul_f64.argtypes = [P, P, i, i, i, i, P, P]
        L.oracle_gemv_2bit_rows.argtypes = [P, P, P, P, P, i, i, P, i, i, i, i, i, i, P, P]
        L.oracle_gemv_nf4_rows.argtypes = [P, P, P, P, i, i, i, i, i, i, P, P]
        L.oracle_dequant_2bit_one.argtypes = [ctypes.c_uint16, i, ctypes.c_uint16]
        L.oracle_dequant_2bit_one.restype = ctypes.c_float
        L.oracle_half_to_float.argtypes = [ctypes.c_uint16]
        L.oracle_half_to_float.restype = ctypes.c_float
        L.oracle_float_to_half.argtypes = [ctypes.c_float]
        L.oracle_float_to_half.restype = ctypes.c_uint16
        L.oracle_float_to_bf16.argtypes = [ctypes.c_float]
        L.oracle_float_to_bf16.restype = ctypes.c_uint16
        _LIB = L
    return _LIB


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


_KIND = {"f16": 1, "bf16": 2}


# ---------------------------------------------------------------------------
# Lloyd-Max codebook (section 2)
# ---------------------------------------------------------------------------

def lloyd_max(samples: np.ndarray, levels: int = 4, iters: int = 200, init=None) -> np.ndarray:
    """Lloyd's iteration for the MSQE-optimal scalar quantizer of `samples`.

    Alternates the two optimality conditions: thresholds at midpoints of adjacent
    levels, and each level at the mean of the samples in its cell.
    """
    x = np.sort(np.asarray(samples, dtype=np.float64))
    c = np.array(init if init is not None else np.quantile(x, (np.arange(levels) + 0.5) / levels), dtype=np.float64)
    for _ in range(iters):
        t = (c[:-1] + c[1:]) / 2.0
        cells = np.searchsorted(x, t)            # cell boundaries in the sorted samples
        edges = np.concatenate([[0], cells, [len(x)]])
        c = np.array([x[edges[i]:edges[i + 1]].mean() for i in range(levels)])
    return c


def quantizer_mse(samples: np.ndarray, levels) -> float:
    """Mean squared error of nearest-level quantization of `samples` to `levels`."""
    x = np.asarray(samples, dtype=np.float64)
    lv = np.asarray(levels, dtype=np.float64)
    q = np.argmin(np.abs(x[:, None] - lv[None, :]), axis=1)
    return float(np.mean((x - lv[q]) ** 2))


def uniform_minmax_mse(samples: np.ndarray, group: int) -> float:
    """MSE of the 4-level linear grid between each group's min and max (the foil of section 2)."""
    x = np.asarray(samples, dtype=np.float64)
    x = x[: len(x) // group * group].reshape(-1, group)
    lo = x.min(axis=1, keepdims=True)
    hi = x.max(axis=1, keepdims=True)
    step = (hi - lo) / 3.0
    q = np.clip(np.rint((x - lo) / np.where(step > 0, step, 1.0)), 0, 3)
    return float(np.mean((x - (lo + q * step)) ** 2))


# ---------------------------------------------------------------------------
# 2-bit quantizer (sections 3 and 4)
# ---------------------------------------------------------------------------

def nearest_centroid(z: np.ndarray) -> np.ndarray:
    """q_i = argmin_k |z_i - C_k|; the lowest index wins a tie."""
    z = np.asarray(z, dtype=np.float64)
    C = np.asarray(CODEBOOK, dtype=np.float64)
    d = np.abs(z[..., None] - C)
    return np.argmin(d, axis=-1).astype(np.uint8)       # argmin returns the first minimum


def _normalise(w: np.ndarray) -> np.ndarray:
    """(w - mean)/std with the population std (ddof=0); all zeros when std == 0."""
    w = np.asarray(w, dtype=np.float64)
    mu = w.mean()
    sd = w.std()
    if sd == 0.0:
        return np.zeros_like(w)
    return (w - mu) / sd


def ols_fit(w: np.ndarray, c: np.ndarray, eps: float = OLS_EPS) -> tuple[float, float]:
    """Closed-form least squares of w ~ S*c + Z (section 3):

    S = sum (w_i - mean w)(c_i - mean c) / (sum (c_i - mean c)^2 + eps),  Z = mean w - S * mean c.
    """
    w = np.asarray(w, dtype=np.float64)
    c = np.asarray(c, dtype=np.float64)
    wb = w.mean()
    cb = c.mean()
    S = float(np.sum((w - wb) * (c - cb)) / (np.sum((c - cb) ** 2) + eps))
    Z = float(wb - S * cb)
    return S, Z


def anchor_count(K: int, frac: float = ANCHOR_FRAC) -> int:
    """floor(frac * K) anchor columns."""
    return int(np.floor(frac * K))


def activation_profile(sigma_c: np.ndarray) -> np.ndarray:
    """mean|X_c| of a zero-mean Gaussian channel with std sigma_c: sqrt(2/pi) * sigma_c."""
    return np.sqrt(2.0 / np.pi) * np.asarray(sigma_c, dtype=np.float64)


def select_anchors(W: np.ndarray, profile: np.ndarray, frac: float = ANCHOR_FRAC) -> np.ndarray:
    """Top floor(frac*K) columns by I_c = ||W[:,c]||_2 * profile_c; ties to the lower column.

    Returns the chosen columns sorted ascending (int32).
    """
    W = np.asarray(W, dtype=np.float64)
    K = W.shape[1]
    A = anchor_count(K, frac)
    score = np.sqrt(np.sum(W * W, axis=0)) * np.asarray(profile, dtype=np.float64)
    order = sorted(range(K), key=lambda c: (-score[c], c))
    return np.sort(np.array(order[:A], dtype=np.int64)).astype(np.int32)


def quantize_2bit(W: np.ndarray, anchor_idx: np.ndarray, lda: int | None = None) -> dict:
    """Quantize W [N][K] to codes, per-group fp16 scale/offset and fp16 anchors.

    For each row and each group of 32 consecutive columns:
      1. V = the non-anchor positions of the group;
      2. z = (W_V - mean W_V) / std W_V (population std; z = 0 if std = 0);
      3. q = nearest centroid of z;
      4. (S, Z) = OLS fit of W_V on C[q];
      5. stored scale/offset = binary16 RNE of S and Z (0 and 0 for an all-anchor group).
    Anchor positions store code 0; their binary16 values go to anchor_w[n][a].
    """
    W = np.asarray(W, dtype=np.float32)
    N, K = W.shape
    assert K % GROUP == 0
    anchor_idx = np.asarray(anchor_idx, dtype=np.int32)
    A = len(anchor_idx)
    lda = int(lda if lda is not None else max(8, (A + 7) // 8 * 8))
    is_anchor = np.zeros(K, dtype=bool)
    is_anchor[anchor_idx] = True
    C = np.asarray(CODEBOOK, dtype=np.float64)

    q = np.zeros((N, K), dtype=np.uint8)
    S = np.zeros((N, K // GROUP), dtype=np.float64)
    Z = np.zeros((N, K // GROUP), dtype=np.float64)
    W64 = W.astype(np.float64)
    for g in range(K // GROUP):
        cols = np.arange(g * GROUP, (g + 1) * GROUP)
        V = cols[~is_anchor[cols]]
        if len(V) == 0:
            continue
        Wg = W64[:, V]                                      # [N][n_V]
        mu = Wg.mean(axis=1, keepdims=True)
        sd = Wg.std(axis=1, keepdims=True)
        z = np.where(sd > 0, (Wg - mu) / np.where(sd > 0, sd, 1.0), 0.0)
        qg = nearest_centroid(z)
        q[:, V] = qg
        c = C[qg]
        cb = c.mean(axis=1, keepdims=True)
        wb = mu
        S[:, g] = (np.sum((Wg - wb) * (c - cb), axis=1) / (np.sum((c - cb) ** 2, axis=1) + OLS_EPS))
        Z[:, g] = wb[:, 0] - S[:, g] * cb[:, 0]
    anchor_w = np.zeros((N, lda), dtype=np.uint16)
    if A:
        anchor_w[:, :A] = W[:, anchor_idx].astype(np.float16).view(np.uint16)
    return dict(codes=pack_2bit(q), q=q, scales=S.astype(np.float16).view(np.uint16),
                offsets=Z.astype(np.float16).view(np.uint16), S=S, Z=Z,
                anchor_idx=anchor_idx, anchor_w=anchor_w, A=A, ld_anchor=lda, N=N, K=K)


def pack_2bit(q: np.ndarray) -> np.ndarray:
    """codes q [N][K] in 0..3 -> bytes [N][K/4]; column 4j+i goes to bits 2i..2i+1 of byte j."""
    q = np.asarray(q, dtype=np.uint8)
    N, K = q.shape
    out = np.zeros((N, K // 4), dtype=np.uint8)
    for i in range(4):
        out |= (q[:, i::4] & 3) << (2 * i)
    return out


def unpack_2bit(codes: np.ndarray) -> np.ndarray:
    """Inverse of pack_2bit."""
    codes = np.asarray(codes, dtype=np.uint8)
    N, KB = codes.shape
    q = np.zeros((N, KB * 4), dtype=np.uint8)
    for i in range(4):
        q[:, i::4] = (codes >> (2 * i)) & 3
    return q


# ---------------------------------------------------------------------------
# NF4 (block 64, fp32 absmax)
# ---------------------------------------------------------------------------

def quantize_nf4(W: np.ndarray) -> dict:
    """Blocks of 64 consecutive weights along K: absmax = max|w| (fp32),
    q = argmin_k |w/absmax - T[k]| (lower index on ties; q = index of 0 if absmax = 0)."""
    W = np.asarray(W, dtype=np.float32)
    N, K = W.shape
    assert K % NF4_BLOCK == 0
    T = nf4_table().astype(np.float64)
    blocks = W.reshape(N, K // NF4_BLOCK, NF4_BLOCK)
    absmax = np.max(np.abs(blocks), axis=2).astype(np.float32)     # exact in fp32
    am = absmax.astype(np.float64)[:, :, None]
    r = np.where(am > 0, blocks.astype(np.float64) / np.where(am > 0, am, 1.0), 0.0)
    q = np.argmin(np.abs(r[..., None] - T), axis=-1).astype(np.uint8).reshape(N, K)
    return dict(codes=pack_nf4(q), q=q, absmax=absmax, N=N, K=K)


def pack_nf4(q: np.ndarray) -> np.ndarray:
    """codes q [N][K] in 0..15 -> bytes [N][K/2]; column 2j low nibble, 2j+1 high nibble."""
    q = np.asarray(q, dtype=np.uint8)
    return ((q[:, 0::2] & 15) | ((q[:, 1::2] & 15) << 4)).astype(np.uint8)


def unpack_nf4(codes: np.ndarray) -> np.ndarray:
    codes = np.asarray(codes, dtype=np.uint8)
    N, KB = codes.shape
    q = np.zeros((N, KB * 2), dtype=np.uint8)
    q[:, 0::2] = codes & 15
    q[:, 1::2] = codes >> 4
    return q


# ---------------------------------------------------------------------------
# v3.2 INT4: uniform symmetric grid, global static permutation, top-1% outliers
# ---------------------------------------------------------------------------

def int4_permutation(W: np.ndarray, profile: np.ndarray) -> np.ndarray:
    """The static column order: input columns by descending impact score
    I_c = ||W[:,c]||_2 * profile_c (the score the v4.0 anchors use), ties to the lower
    column.  perm[j] is the column stored at permuted position j (int32)."""
    W = np.asarray(W, dtype=np.float64)
    K = W.shape[1]
    score = np.sqrt(np.sum(W * W, axis=0)) * np.asarray(profile, dtype=np.float64)
    return np.array(sorted(range(K), key=lambda c: (-score[c], c)), dtype=np.int32)


def quantize_int4(W: np.ndarray, perm: np.ndarray, anchor_idx: np.ndarray, lda: int | None = None) -> dict:
    """Quantize W [N][K] to the INT4 format.

    Columns are taken in the order perm; each row's permuted positions form groups of 32.
    For a group with V = its non-anchor positions:
      S = max |W_V| / 7 (fp64), stored as binary16 (RNE);
      q = clamp(round_half_even(W / S16), -7, 7) with the stored S16 (q = 0 when S16 = 0);
    anchor positions store q = 0 (exactly 0 on the zero-point-0 grid); their binary16
    values go to anchor_w[n][a] for the ascending anchor_idx.
    """
    W = np.asarray(W, dtype=np.float32)
    N, K = W.shape
    assert K % INT4_GROUP == 0
    perm = np.asarray(perm, dtype=np.int32)
    anchor_idx = np.asarray(anchor_idx, dtype=np.int32)
    A = len(anchor_idx)
    lda = int(lda if lda is not None else max(8, (A + 7) // 8 * 8))
    is_anchor = np.zeros(K, dtype=bool)
    is_anchor[anchor_idx] = True
    Wp = W[:, perm].astype(np.float64)                 # permuted columns
    anchor_p = is_anchor[perm]
    q = np.zeros((N, K), dtype=np.int8)
    S16 = np.zeros((N, K // INT4_GROUP), dtype=np.float16)
    for g in range(K // INT4_GROUP):
        pos = np.arange(g * INT4_GROUP, (g + 1) * INT4_GROUP)
        V = pos[~anchor_p[pos]]
        if len(V) == 0:
            continue
        absmax = np.max(np.abs(Wp[:, V]), axis=1)
        s16 = (absmax / INT4_QMAX).astype(np.float16)       # float64 -> binary16, RNE
        S16[:, g] = s16
        s = s16.astype(np.float64)[:, None]
        r = np.where(s > 0, Wp[:, V] / np.where(s > 0, s, 1.0), 0.0)
        q[:, V] = np.clip(np.rint(r), -INT4_QMAX, INT4_QMAX).astype(np.int8)
    anchor_w = np.zeros((N, lda), dtype=np.uint16)
    if A:
        anchor_w[:, :A] = W[:, anchor_idx].astype(np.float16).view(np.uint16)
    return dict(codes=pack_int4(q), q=q, scales=S16.view(np.uint16), perm=perm, anchor_idx=anchor_idx,
                anchor_w=anchor_w, A=A, ld_anchor=lda, N=N, K=K)


def pack_int4(q: np.ndarray) -> np.ndarray:
    """signed codes q [N][K] in -8..7 -> bytes [N][K/2]: position 2j in the low nibble, 2j+1 in the
    high nibble, each as 4-bit two's complement."""
    u = (np.asarray(q, dtype=np.int16) & 15).astype(np.uint8)
    return (u[:, 0::2] | (u[:, 1::2] << 4)).astype(np.uint8)


def unpack_int4(codes: np.ndarray) -> np.ndarray:
    u = unpack_nf4(codes).astype(np.int16)
    return np.where(u >= 8, u - 16, u).astype(np.int8)


def dequant_int4(p: dict) -> np.ndarray:
    """fp32 W_eff [N][K] in original column order: S * q at column perm[j], anchors substituted."""
    L = _lib()
    N, K, A = int(p["N"]), int(p["K"]), int(p["A"])
    out = np.empty((N, K), dtype=np.float32)
    L.oracle_dequant_int4(_p(np.ascontiguousarray(p["codes"], dtype=np.uint8)),
                          _p(np.ascontiguousarray(p["scales"], dtype=np.uint16)),
                          _p(np.ascontiguousarray(p["perm"], dtype=np.int32)),
                          _p(np.ascontiguousarray(p["anchor_idx"], dtype=np.int32)),
                          _p(np.ascontiguousarray(p["anchor_w"], dtype=np.uint16)), A, int(p["ld_anchor"]), N, K,
                          _p(out))
    return out


# ---------------------------------------------------------------------------
# Dequantization and reference products (compiled C)
# ---------------------------------------------------------------------------

def dequant_2bit(p: dict) -> np.ndarray:
    """fp32 W_eff [N][K]: fmaf(S, C[q], Z) per weight, anchor columns replaced by their fp16 values."""
    L = _lib()
    N, K, A = int(p["N"]), int(p["K"]), int(p["A"])
    codes = np.ascontiguousarray(p["codes"], dtype=np.uint8)
    sc = np.ascontiguousarray(p["scales"], dtype=np.uint16)
    of = np.ascontiguousarray(p["offsets"], dtype=np.uint16)
    ai = np.ascontiguousarray(p["anchor_idx"], dtype=np.int32)
    aw = np.ascontiguousarray(p["anchor_w"], dtype=np.uint16)
    out = np.empty((N, K), dtype=np.float32)
    L.oracle_dequant_2bit(_p(codes), _p(sc), _p(of), _p(ai), _p(aw), A, int(p["ld_anchor"]), N, K, _p(out))
    return out


def dequant_nf4(p: dict) -> np.ndarray:
    """fp32 W_eff [N][K] = T[q] * absmax (one fp32 rounding)."""
    L = _lib()
    N, K = int(p["N"]), int(p["K"])
    codes = np.ascontiguousarray(p["codes"], dtype=np.uint8)
    am = np.ascontiguousarray(p["absmax"], dtype=np.float32)
    T = nf4_table()
    out = np.empty((N, K), dtype=np.float32)
    L.oracle_dequant_nf4(_p(codes), _p(am), _p(T), N, K, _p(out))
    return out


# ---------------------------------------------------------------------------
# NF4 with double quantization (QLoRA): the block maxima stored as 8-bit floats
# ---------------------------------------------------------------------------

NF4_DQ_BLOCK = 256          # first-level constants per second-level block


def e4m3_decode(codes) -> np.ndarray:
    """8-bit float (E4M3) codes -> float64 values (NaN for 0x7F / 0xFF)."""
    L = _lib()
    c = np.asarray(codes, dtype=np.uint8)
    return np.array([L.oracle_e4m3_to_double(int(v)) for v in c.ravel()], dtype=np.float64).reshape(c.shape)


def e4m3_encode(values) -> np.ndarray:
    """float64 values -> nearest E4M3 codes (ties to the even mantissa), saturating at +-448."""
    L = _lib()
    v = np.asarray(values, dtype=np.float64)
    return np.array([L.oracle_double_to_e4m3(float(x)) for x in v.ravel()], dtype=np.uint8).reshape(v.shape)


def double_quantize_absmax(absmax: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """The second quantization of the fp32 block maxima c [N][K/64].

    mean = the mean of all c (fp64, rounded once to fp32); in row-major order, each run of 256
    consecutive c (the last may be shorter) is block j with s2_j = max |c - mean| / 448 (fp64,
    rounded once to fp32); acode_i = E4M3((c_i - mean) / s2_j) from the fp64 quotient (0 when
    s2_j = 0).  Returns (acodes uint8 [N][K/64], second float32 [1 + blocks] = [mean, s2_0, ...]).
    """
    c = np.asarray(absmax, dtype=np.float32)
    flat = c.ravel().astype(np.float64)
    mean32 = np.float32(np.sum(flat) / flat.size)
    nb = (flat.size + NF4_DQ_BLOCK - 1) // NF4_DQ_BLOCK
    s2 = np.zeros(nb, dtype=np.float32)
    codes = np.zeros(flat.size, dtype=np.uint8)
    for j in range(nb):
        seg = flat[j * NF4_DQ_BLOCK:(j + 1) * NF4_DQ_BLOCK] - np.float64(mean32)
        s2[j] = np.float32(np.max(np.abs(seg)) / 448.0)
        if s2[j] > 0:
            codes[j * NF4_DQ_BLOCK:j * NF4_DQ_BLOCK + len(seg)] = e4m3_encode(seg / np.float64(s2[j]))
    return codes.reshape(c.shape), np.concatenate([[mean32], s2]).astype(np.float32)


def quantize_nf4_dq(W: np.ndarray) -> dict:
    """NF4 codes from the fp32 block maxima (exactly as quantize_nf4), then the maxima
    double-quantized.  Storage: codes [N][K/2], acodes uint8 [N][K/64], second fp32."""
    p = quantize_nf4(W)
    acodes, second = double_quantize_absmax(p["absmax"])
    return dict(codes=p["codes"], q=p["q"], absmax=p["absmax"], acodes=acodes, second=second, N=p["N"], K=p["K"])


def dequant_nf4_dq(p: dict) -> np.ndarray:
    """fp32 W_eff [N][K] = T[q] * c', c' = fmaf(E4M3(acode), s2, mean) (one fp32 rounding each)."""
    L = _lib()
    N, K = int(p["N"]), int(p["K"])
    out = np.empty((N, K), dtype=np.float32)
    L.oracle_dequant_nf4_dq(_p(np.ascontiguousarray(p["codes"], dtype=np.uint8)),
                            _p(np.ascontiguousarray(p["acodes"], dtype=np.uint8)),
                            _p(np.ascontiguousarray(p["second"], dtype=np.float32)), _p(nf4_table()), N, K, _p(out))
    return out


def round_to(w32: np.ndarray, dtype: str) -> np.ndarray:
    """fp32 -> 'f16' / 'bf16' bit patterns (RNE), or the fp32 array itself for 'f32'."""
    w32 = np.ascontiguousarray(w32, dtype=np.float32)
    if dtype == "f32":
        return w32
    out = np.empty(w32.shape, dtype=np.uint16)
    _lib().oracle_round_f32(_p(w32), w32.size, _KIND[dtype], _p(out))
    return out


def matmul_ref(W_eff: np.ndarray, x_bits: np.ndarray, x_dtype: str) -> tuple[np.ndarray, np.ndarray]:
    """y[m][n] = sum_k W_eff[n][k] x[m][k] and E[m][n] = sum_k |W_eff[n][k]| |x[m][k]|, in fp64."""
    W = np.ascontiguousarray(W_eff, dtype=np.float32)
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    N, K = W.shape
    M = x.shape[0]
    y = np.empty((M, N), dtype=np.float64)
    E = np.empty((M, N), dtype=np.float64)
    _lib().oracle_matmul_f64(_p(W), _p(x), _KIND[x_dtype], M, N, K, _p(y), _p(E))
    return y, E


def gemv_2bit_rows(p: dict, x_bits: np.ndarray, x_dtype: str, n0: int, n1: int) -> np.ndarray:
    """fp64 y[:, n0:n1] for a 2-bit matrix, row by row (sampled checks, CPU baseline)."""
    L = _lib()
    N, K, A = int(p["N"]), int(p["K"]), int(p["A"])
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    M = x.shape[0]
    y = np.empty((M, n1 - n0), dtype=np.float64)
    scratch = np.empty(K, dtype=np.float32)
    L.oracle_gemv_2bit_rows(_p(np.ascontiguousarray(p["codes"])), _p(np.ascontiguousarray(p["scales"])),
                            _p(np.ascontiguousarray(p["offsets"])), _p(np.ascontiguousarray(p["anchor_idx"], dtype=np.int32)),
                            _p(np.ascontiguousarray(p["anchor_w"])), A, int(p["ld_anchor"]), _p(x), _KIND[x_dtype],
                            M, N, K, int(n0), int(n1), _p(scratch), _p(y))
    return y


def gemv_nf4_rows(p: dict, x_bits: np.ndarray, x_dtype: str, n0: int, n1: int) -> np.ndarray:
    L = _lib()
    N, K = int(p["N"]), int(p["K"])
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    M = x.shape[0]
    y = np.empty((M, n1 - n0), dtype=np.float64)
    scratch = np.empty(K, dtype=np.float32)
    T = nf4_table()
    L.oracle_gemv_nf4_rows(_p(np.ascontiguousarray(p["codes"])), _p(np.ascontiguousarray(p["absmax"], dtype=np.float32)),
                           _p(T), _p(x), _KIND[x_dtype], M, N, K, int(n0), int(n1), _p(scratch), _p(y))
    return y


def row_error_scale(W_rows: np.ndarray, x_bits: np.ndarray, x_dtype: str) -> np.ndarray:
    """E[m][n] = sum_k |x[m][k]| |W[n][k]| for a few dequantized rows (fp64)."""
    return np.abs(x_values(x_bits, x_dtype)) @ np.abs(np.asarray(W_rows, dtype=np.float64)).T


def x_values(x_bits: np.ndarray, x_dtype: str) -> np.ndarray:
    """16-bit x bit patterns -> fp64 values (vectorised, exact)."""
    b = np.ascontiguousarray(x_bits, dtype=np.uint16)
    if x_dtype == "f16":
        return b.view(np.float16).astype(np.float64)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
