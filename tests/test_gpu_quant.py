"""GPU parity of the quantizers (lq_select_anchors, lq_quantize_2bit, lq_quantize_nf4)
against the CPU oracle's quantizers.

Every output is integer or a binary16/fp32 bit pattern, and both sides take each
floating-point decision in fp64 with the same operations and summation order, so
the comparison is bit for bit: anchor columns, packed codes, scale/offset bits,
anchor weights, NF4 codes and absmax.
"""
import numpy as np
import pytest

import synth
from oracle import oracle as O

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lqm():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import bit_weight_quantized_dequant_gb300 as lq
    lq.build()
    return lq


@pytest.fixture(scope="module")
def handle(lqm):
    h = lqm.Handle(0)
    yield h
    h.close()


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def check_2bit(gpu, ref, rows=None):
    """Compare a device QuantWeights with an oracle dict (optionally only `rows` of the device one)."""
    sel = slice(None) if rows is None else rows
    assert np.array_equal(gpu.codes.cpu().numpy()[sel], ref["codes"]), "codes"
    assert np.array_equal(gpu.scales.cpu().view(torch.int16).numpy().view(np.uint16)[sel], ref["scales"]), "scale bits"
    assert np.array_equal(gpu.offsets.cpu().view(torch.int16).numpy().view(np.uint16)[sel], ref["offsets"]), "offset bits"
    if ref["A"] > 0:
        aw = gpu.anchor_w.cpu().view(torch.int16).numpy().view(np.uint16)[sel]
        assert np.array_equal(aw, ref["anchor_w"]), "anchor_w bits"
    else:
        assert gpu.anchor_w is None


@pytest.mark.parametrize("N,K,outlier_frac", [(512, 256, 0.0), (300, 4096, 0.01), (64, 11008, 0.01), (33, 8192, 0.01)])
def test_select_anchors_matches_oracle(lqm, handle, N, K, outlier_frac):
    W = synth.weights(N, K, 0.02, seed=11, cfg=2, matrix_id=K)
    outl = synth.outlier_channels(K, outlier_frac, seed=11, cfg=2)
    prof = O.activation_profile(synth.channel_sigma(K, outl, 20.0))
    ref = O.select_anchors(W, prof)
    got = handle.select_anchors(dev(W), profile=dev(prof)).cpu().numpy()
    assert got.dtype == np.int32 and len(got) == O.anchor_count(K)
    assert np.array_equal(got, ref)
    assert set(outl.tolist()) <= set(got.tolist())      # every x20 channel is an anchor


def test_select_anchors_ties_go_to_the_lower_column(lqm, handle):
    """Duplicate columns give equal scores; the lower column wins, in the oracle and on the GPU."""
    N, K = 40, 320
    W = synth.weights(N, K, 0.02, seed=3)
    W[:, 200:] = W[:, 0:120]            # columns 200.. copy 0..119: every score appears twice
    ref = O.select_anchors(W, np.ones(K))
    got = handle.select_anchors(dev(W)).cpu().numpy()
    assert np.array_equal(got, ref)
    # A = K takes every column; A = 1 the single largest
    assert np.array_equal(handle.select_anchors(dev(W), A=K).cpu().numpy(), np.arange(K, dtype=np.int32))
    score = np.sqrt((W.astype(np.float64) ** 2).sum(axis=0))
    assert handle.select_anchors(dev(W), A=1).cpu().numpy().tolist() == [int(np.flatnonzero(score == score.max())[0])]


@pytest.mark.parametrize("N,K", [(512, 256), (200, 4096), (48, 11008)])
def test_quantize_2bit_bit_exact(lqm, handle, N, K):
    W = synth.weights(N, K, 0.02, seed=5, cfg=2, matrix_id=N)
    outl = synth.outlier_channels(K, 0.01, seed=5, cfg=2)
    ai = O.select_anchors(W, O.activation_profile(synth.channel_sigma(K, outl, 20.0)))
    ref = O.quantize_2bit(W, ai)
    got = handle.quantize_2bit(dev(W), dev(ai))
    torch.cuda.synchronize()
    check_2bit(got, ref)


def test_quantize_2bit_degenerate_groups(lqm, handle):
    """All-anchor group, groups with 1 and 7 non-anchor values (the short-sum branch), a
    constant group (std 0), a zero row, and a group with anchors at both ends."""
    N, K = 6, 128
    W = synth.weights(N, K, 0.02, seed=9)
    W[2, 64:96] = 0.013                     # constant group: z = 0, every code 1
    W[3, :] = 0.0                           # zero row
    anchors = list(range(0, 32))            # group 0: all anchors
    anchors += [c for c in range(32, 64) if c != 40]            # group 1: one value left
    anchors += [c for c in range(96, 128) if c not in (97, 101, 103, 110, 111, 120, 125)]   # group 3: seven left
    anchors += [64, 95]                      # group 2: anchors at both ends
    ai = np.array(sorted(anchors), dtype=np.int32)
    ref = O.quantize_2bit(W, ai)
    got = handle.quantize_2bit(dev(W), dev(ai))
    torch.cuda.synchronize()
    check_2bit(got, ref)
    assert np.all(ref["scales"][:, 0] == 0) and np.all(ref["offsets"][:, 0] == 0)


def test_quantize_2bit_without_anchors(lqm, handle):
    W = synth.weights(96, 512, 0.02, seed=21)
    half = np.arange(16, dtype=np.float32) / 256          # dyadic values: every sum is exact
    W[0, :32] = np.concatenate([half, -half])               # mean exactly 0 and one value equal to it (z = 0)
    ref = O.quantize_2bit(W, np.zeros(0, np.int32))
    got = handle.quantize_2bit(dev(W))
    torch.cuda.synchronize()
    check_2bit(got, ref)


def test_quantize_then_dequant_and_gemv(lqm, handle):
    """GPU-quantized weights feed the hot path: dequant equals the oracle's, and gemv meets its bound."""
    N, K = 256, 2048
    W = synth.weights(N, K, 0.02, seed=4)
    outl = synth.outlier_channels(K, 0.01, seed=4)
    prof = O.activation_profile(synth.channel_sigma(K, outl, 20.0))
    Wd = dev(W)
    ai = handle.select_anchors(Wd, profile=dev(prof))
    w = handle.quantize_2bit(Wd, ai)
    ref = O.quantize_2bit(W, O.select_anchors(W, prof))
    deq = handle.dequant(w).cpu().numpy()
    assert np.array_equal(deq.view(np.uint32), O.dequant_2bit(ref).view(np.uint32))
    xb = synth.activations(1, K, "f16", synth.channel_sigma(K, outl, 20.0), seed=4)
    y = handle.gemv(w, torch.from_numpy(xb).view(torch.float16).cuda()).cpu().numpy()
    yref, E = O.matmul_ref(O.dequant_2bit(ref), xb, "f16")
    assert np.all(np.abs(y - yref) <= 1e-3 * E + 1e-30)


@pytest.mark.parametrize("N,K", [(64, 256), (300, 4096), (16, 11008)])
def test_quantize_nf4_bit_exact(lqm, handle, N, K):
    W = synth.weights(N, K, 0.02, seed=7, cfg=3, matrix_id=K, big_frac=0.001, big_mult=10.0)
    W[1, 64:128] = 0.0                        # absmax 0: every code is the index of level 0
    T = O.nf4_table()
    mids = ((T[:-1].astype(np.float64) + T[1:]) / 2).astype(np.float32)
    W[2, :64] = np.concatenate([[1.0], T, mids, -mids, 0.5 * T, [0.0]])   # levels, (near-)midpoints; absmax 1
    ref = O.quantize_nf4(W)
    got = handle.quantize_nf4(dev(W))
    torch.cuda.synchronize()
    assert np.array_equal(got.codes.cpu().numpy(), ref["codes"])
    assert np.array_equal(got.scales.cpu().numpy().view(np.uint32), ref["absmax"].view(np.uint32))


def test_quantizers_14b_layer_sampled(lqm, handle):
    """Full-size 14B gate projection (13824 x 5120): anchors over all rows, codes on sampled rows."""
    N, K = 13824, 5120
    W = synth.weights(N, K, 0.02, seed=8, cfg=5, matrix_id=1)
    outl = synth.outlier_channels(K, 0.01, seed=8, cfg=5)
    prof = O.activation_profile(synth.channel_sigma(K, outl, 20.0))
    Wd = dev(W)
    ai = handle.select_anchors(Wd, profile=dev(prof))
    ai_ref = O.select_anchors(W, prof)
    assert np.array_equal(ai.cpu().numpy(), ai_ref)
    w = handle.quantize_2bit(Wd, ai)
    rows = np.sort(np.random.default_rng(8).choice(N, 64, replace=False))
    rows = np.unique(np.concatenate([rows, [0, N - 1]]))
    check_2bit(w, O.quantize_2bit(W[rows], ai_ref), rows=rows)
    wn = handle.quantize_nf4(Wd)
    refn = O.quantize_nf4(W[rows])
    assert np.array_equal(wn.codes.cpu().numpy()[rows], refn["codes"])
    assert np.array_equal(wn.scales.cpu().numpy()[rows].view(np.uint32), refn["absmax"].view(np.uint32))
