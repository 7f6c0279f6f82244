"""Seeded synthetic inputs for the low-bit linear layer (dequantize-and-multiply).

This module only draws random numbers and lays them out; it holds no step of the
quantization or dequantization method.  Tests, the benchmark and the oracle all
take their inputs from here, so the GPU path and the CPU oracle see identical
bytes.

Workloads stand in for the decoder layers that the otf-llm 4.0.1 README benchmarks
("Performance Benchmark" table: Qwen2.5-3B..32B) and for the 70B layers that the
AutoBot-AI #1946 issue streams ("Background"): there are no checkpoints here, so
weights are Gaussian draws with the stated standard deviations.

Random streams are keyed by (seed, workload id, matrix id) through NumPy's
SeedSequence, so any single matrix can be regenerated on its own.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "rng", "weights", "outlier_channels", "channel_sigma", "activations",
    "f32_to_f16_bits", "f32_to_bf16_bits", "bits_to_f32",
    "random_packed_2bit", "random_packed_nf4", "random_packed_2bit_sets", "LAYER_SHAPES",
]

# (name, N_out, K_in) per decoder layer, the shapes of the workload table.
LAYER_SHAPES = {
    "7b": [("q", 4096, 4096), ("k", 4096, 4096), ("v", 4096, 4096), ("o", 4096, 4096),
           ("gate", 11008, 4096), ("up", 11008, 4096), ("down", 4096, 11008)],
    "70b": [("q", 8192, 8192), ("k", 1024, 8192), ("v", 1024, 8192), ("o", 8192, 8192),
            ("gate", 28672, 8192), ("up", 28672, 8192), ("down", 8192, 28672)],
    "14b": [("q", 5120, 5120), ("k", 5120, 5120), ("v", 5120, 5120), ("o", 5120, 5120),
            ("gate", 13824, 5120), ("up", 13824, 5120), ("down", 5120, 13824)],
}


def rng(seed: int, cfg: int = 0, matrix_id: int = 0) -> np.random.Generator:
    """Independent generator for one (seed, workload, matrix) triple."""
    return np.random.default_rng(np.random.SeedSequence([int(seed), int(cfg), int(matrix_id)]))


def weights(N: int, K: int, sigma: float, seed: int = 0, cfg: int = 0, matrix_id: int = 0,
            big_frac: float = 0.0, big_mult: float = 10.0) -> np.ndarray:
    """W ~ N(0, sigma^2) as float32 [N][K] (out x in).

    With big_frac > 0, floor(big_frac*N*K) entries chosen uniformly without
    replacement are multiplied by big_mult (the "0.1% entries x10" workload).
    """
    g = rng(seed, cfg, matrix_id)
    W = (g.standard_normal((N, K), dtype=np.float32) * np.float32(sigma)).astype(np.float32)
    n_big = int(np.floor(big_frac * N * K))
    if n_big > 0:
        flat = g.choice(N * K, size=n_big, replace=False)
        W.reshape(-1)[flat] *= np.float32(big_mult)
    return W


def outlier_channels(K: int, frac: float = 0.01, seed: int = 0, cfg: int = 0) -> np.ndarray:
    """floor(frac*K) input channels, chosen by seed, sorted ascending (int64)."""
    n = int(np.floor(frac * K))
    if n == 0:
        return np.zeros(0, dtype=np.int64)
    g = rng(seed, cfg, 10_000)
    return np.sort(g.choice(K, size=n, replace=False)).astype(np.int64)


def channel_sigma(K: int, outliers: np.ndarray, mult: float = 20.0) -> np.ndarray:
    """Per-input-channel standard deviation of x: 1 everywhere, `mult` on outliers."""
    s = np.ones(K, dtype=np.float64)
    s[np.asarray(outliers, dtype=np.int64)] = mult
    return s


def f32_to_f16_bits(a: np.ndarray) -> np.ndarray:
    """float32/float64 -> IEEE binary16 bit patterns (uint16), round to nearest even."""
    return np.asarray(a).astype(np.float16).view(np.uint16)


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 bit patterns (uint16), round to nearest even (no NaNs expected)."""
    u = np.ascontiguousarray(np.asarray(a, dtype=np.float32)).view(np.uint32).astype(np.uint64)
    bias = np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))
    return ((u + bias) >> np.uint64(16)).astype(np.uint16)


def bits_to_f32(bits: np.ndarray, dtype: str) -> np.ndarray:
    """uint16 bit patterns of 'f16' or 'bf16' -> exact float32 values."""
    bits = np.asarray(bits, dtype=np.uint16)
    if dtype == "f16":
        return bits.view(np.float16).astype(np.float32)
    if dtype == "bf16":
        return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)
    raise ValueError(dtype)


def activations(M: int, K: int, dtype: str = "f16", sigma_c: np.ndarray | None = None,
                seed: int = 0, cfg: int = 0, matrix_id: int = 0) -> np.ndarray:
    """x ~ N(0, sigma_c^2) per channel, rounded to `dtype`; returns uint16 bits [M][K]."""
    g = rng(seed, cfg, 20_000 + matrix_id)
    x = g.standard_normal((M, K), dtype=np.float32)
    if sigma_c is not None:
        x = (x * np.asarray(sigma_c, dtype=np.float32)[None, :]).astype(np.float32)
    return f32_to_f16_bits(x) if dtype == "f16" else f32_to_bf16_bits(x)


def random_packed_2bit(N: int, K: int, A: int, sigma: float = 0.02, seed: int = 0, cfg: int = 0,
                       matrix_id: int = 0, ld_anchor: int | None = None) -> dict:
    """Random bytes in the 2-bit storage layout, for throughput runs at full size.

    codes: uniform random bytes [N][K/4]; scales ~ sigma*U(0.8, 1.2) and offsets ~
    N(0, sigma^2/32) rounded to binary16 [N][K/32]; anchor_idx: A distinct sorted
    columns; anchor_w ~ N(0, sigma^2) binary16 [N][ld_anchor], zero past A.
    No quantizer runs here: these are draws of the right sizes and magnitudes.
    """
    g = rng(seed, cfg, 30_000 + matrix_id)
    ld = int(ld_anchor if ld_anchor is not None else max(8, (A + 7) // 8 * 8))
    codes = g.integers(0, 256, size=(N, K // 4), dtype=np.uint8)
    scales = f32_to_f16_bits(sigma * g.uniform(0.8, 1.2, size=(N, K // 32)).astype(np.float32))
    offsets = f32_to_f16_bits((sigma / np.sqrt(32.0)) * g.standard_normal((N, K // 32)).astype(np.float32))
    anchor_idx = np.sort(g.choice(K, size=A, replace=False)).astype(np.int32) if A > 0 else np.zeros(0, np.int32)
    aw = np.zeros((N, ld), dtype=np.float32)
    if A > 0:
        aw[:, :A] = sigma * g.standard_normal((N, A)).astype(np.float32)
    anchor_w = f32_to_f16_bits(aw)
    if A > 0:
        anchor_w[:, A:] = 0
    return dict(codes=codes, scales=scales, offsets=offsets, anchor_idx=anchor_idx,
                anchor_w=anchor_w, A=A, ld_anchor=ld, N=N, K=K)


def random_packed_nf4(N: int, K: int, sigma: float = 0.02, seed: int = 0, cfg: int = 0,
                      matrix_id: int = 0) -> dict:
    """Random bytes in the NF4 storage layout: codes [N][K/2], absmax float32 [N][K/64]."""
    g = rng(seed, cfg, 40_000 + matrix_id)
    codes = g.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    absmax = (sigma * g.uniform(2.0, 4.0, size=(N, K // 64))).astype(np.float32)
    return dict(codes=codes, absmax=absmax, N=N, K=K)


def random_packed_int4(N: int, K: int, A: int, sigma: float = 0.02, seed: int = 0, cfg: int = 0,
                       matrix_id: int = 0) -> dict:
    """Random bytes in the INT4 storage layout, for runs at full size.

    perm: a random permutation of the K columns (int32); codes: random bytes [N][K/2]
    with the nibbles of the permuted positions that hold an anchor column set to 0 (the
    layout stores code 0 there); scales ~ (sigma/4)*U(0.8, 1.2) as binary16 [N][K/32];
    anchor_idx: A distinct sorted columns; anchor_w ~ N(0, sigma^2) binary16, zero past A.
    """
    g = rng(seed, cfg, 60_000 + matrix_id)
    ld = max(8, (A + 7) // 8 * 8)
    perm = g.permutation(K).astype(np.int32)
    codes = g.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    anchor_idx = np.sort(g.choice(K, size=A, replace=False)).astype(np.int32) if A > 0 else np.zeros(0, np.int32)
    if A > 0:
        pos = np.flatnonzero(np.isin(perm, anchor_idx))          # permuted positions of anchor columns
        keep = np.where(pos % 2 == 0, 0xF0, 0x0F).astype(np.uint8)
        for j, m in zip(pos // 2, keep):
            codes[:, j] &= m
    scales = f32_to_f16_bits((sigma / 4) * g.uniform(0.8, 1.2, size=(N, K // 32)).astype(np.float32))
    anchor_w = np.zeros((N, ld), dtype=np.uint16)
    if A > 0:
        anchor_w[:, :A] = f32_to_f16_bits(sigma * g.standard_normal((N, A)).astype(np.float32))
    return dict(codes=codes, scales=scales, perm=perm, anchor_idx=anchor_idx, anchor_w=anchor_w,
                A=A, ld_anchor=ld, N=N, K=K)


def random_packed_nf4_dq(N: int, K: int, sigma: float = 0.02, seed: int = 0, cfg: int = 0,
                         matrix_id: int = 0) -> dict:
    """Random bytes in the double-quantized NF4 layout: codes [N][K/2]; acodes uint8 [N][K/64]
    (8-bit float codes of either sign, the two NaN codes excluded); second = [mean, s2_0, ...]
    float32 with mean ~ 3 sigma and s2 ~ sigma * U(0.5, 1) / 448."""
    g = rng(seed, cfg, 70_000 + matrix_id)
    codes = g.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    acodes = (g.integers(0, 0x7F, size=(N, K // 64)) | (g.integers(0, 2, size=(N, K // 64)) << 7)).astype(np.uint8)
    nb = (N * (K // 64) + 255) // 256
    second = np.concatenate([[3 * sigma], sigma * g.uniform(0.5, 1.0, nb) / 448.0]).astype(np.float32)
    return dict(codes=codes, acodes=acodes, second=second, N=N, K=K)


def random_packed_2bit_sets(L: int, N: int, K: int, A: int, sigma: float = 0.02, seed: int = 0, cfg: int = 0) -> dict:
    """L independent weight sets of one shape in the 2-bit storage layout, stacked on a
    leading axis (codes [L][N][K/4], scales/offsets [L][N][K/32], anchor_idx [L][A],
    anchor_w [L][N][ld_anchor]); random draws of the right sizes and magnitudes."""
    g = rng(seed, cfg, 50_000)
    ld = max(8, (A + 7) // 8 * 8)
    # codes: a random block of up to 1024 sets, tiled with a distinct XOR byte per tile (every set
    # differs; drawing the full size byte by byte takes tens of seconds)
    T = min(L, 1024)
    base = g.integers(0, 2**32, size=T * N * (K // 4) // 4, dtype=np.uint32).view(np.uint8).reshape(T, N, K // 4)
    codes = np.empty((L, N, K // 4), dtype=np.uint8)
    for i in range(0, L, T):
        n = min(T, L - i)
        np.bitwise_xor(base[:n], np.uint8(((i // T) * 0x9D) & 0xFF), out=codes[i:i + n])
    scales = f32_to_f16_bits(sigma * (np.float32(0.8) + np.float32(0.4) * g.random((L, N, K // 32), dtype=np.float32)))
    offsets = f32_to_f16_bits(np.float32(sigma / np.sqrt(32.0)) * g.standard_normal((L, N, K // 32), dtype=np.float32))
    # A distinct sorted columns per set: the A smallest of K random keys
    keys = g.random((L, K), dtype=np.float32)
    anchor_idx = np.sort(np.argpartition(keys, A, axis=1)[:, :A], axis=1).astype(np.int32)
    anchor_w = np.zeros((L, N, ld), dtype=np.uint16)
    anchor_w[:, :, :A] = f32_to_f16_bits(np.float32(sigma) * g.standard_normal((L, N, A), dtype=np.float32))
    return dict(codes=codes, scales=scales, offsets=offsets, anchor_idx=anchor_idx, anchor_w=anchor_w,
                A=A, ld_anchor=ld, N=N, K=K, L=L)
