"""Helpers shared by the tests: building problems with the oracle and checking bounds."""
from __future__ import annotations

import numpy as np

import synth
from oracle import oracle as O


def quantized_2bit(N, K, seed=0, cfg=0, mid=0, sigma=0.02, outlier_frac=0.01, outlier_mult=20.0):
    """Synthetic W quantized by the oracle (profile-guided anchors, 2-bit G=32)."""
    W = synth.weights(N, K, sigma, seed=seed, cfg=cfg, matrix_id=mid)
    outl = synth.outlier_channels(K, outlier_frac, seed=seed, cfg=cfg)
    prof = O.activation_profile(synth.channel_sigma(K, outl, outlier_mult))
    ai = O.select_anchors(W, prof)
    p = O.quantize_2bit(W, ai)
    return p, outl


def quantized_nf4(N, K, seed=0, cfg=0, mid=0, sigma=0.02, big_frac=0.001):
    W = synth.weights(N, K, sigma, seed=seed, cfg=cfg, matrix_id=mid, big_frac=big_frac, big_mult=10.0)
    return O.quantize_nf4(W)


def x_for(M, K, dtype, outl=None, seed=0, cfg=0, mid=0):
    sig = synth.channel_sigma(K, outl if outl is not None else np.zeros(0, np.int64), 20.0)
    return synth.activations(M, K, dtype, sig, seed=seed, cfg=cfg, matrix_id=mid)


def assert_within(y_gpu: np.ndarray, y_ref: np.ndarray, E: np.ndarray, rel: float, what: str = ""):
    """|y - y_ref| <= rel * E elementwise (E = sum |W_eff||x|)."""
    y_gpu = np.asarray(y_gpu, dtype=np.float64)
    err = np.abs(y_gpu - y_ref)
    bound = rel * E + 1e-30
    bad = err > bound
    if np.any(bad):
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} outputs out of bound; first at {tuple(i)}: "
                             f"gpu={y_gpu[tuple(i)]!r} ref={y_ref[tuple(i)]!r} E={E[tuple(i)]!r} "
                             f"max err/E={np.max(err / (E + 1e-30)):.3e}")
    return float(np.max(err / (E + 1e-30)))


def quantized_int4(N, K, seed=0, cfg=0, mid=0, sigma=0.02, outlier_frac=0.01, outlier_mult=20.0):
    """Synthetic W quantized by the oracle to the INT4 format: the impact-score permutation
    and the top-1% binary16 outlier columns both from the activation profile."""
    W = synth.weights(N, K, sigma, seed=seed, cfg=cfg, matrix_id=mid, big_frac=0.001, big_mult=10.0)
    outl = synth.outlier_channels(K, outlier_frac, seed=seed, cfg=cfg)
    prof = O.activation_profile(synth.channel_sigma(K, outl, outlier_mult))
    perm = O.int4_permutation(W, prof)
    ai = O.select_anchors(W, prof, frac=O.INT4_OUTLIER_FRAC)
    return O.quantize_int4(W, perm, ai), outl
