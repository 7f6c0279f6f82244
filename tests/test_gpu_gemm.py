"""GPU parity of lq_gemm (tcgen05 tensor-core prefill GEMM) against the CPU oracle.

bf16 x: |y - y_ref| <= 4e-3 * sum_k |W_eff||x| (weights rounded once to bf16);
binary16 x: <= 1e-3 * sum_k |W_eff||x|.  Shapes span several 128-row x 256-token
tiles with ragged edges, anchors that split K-blocks, and the 14B-layer prefill
at M = 2048 on sampled rows.
"""
import numpy as np
import pytest

import synth
from oracle import oracle as O
from tests._util import assert_within, quantized_2bit, quantized_nf4, x_for

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

TOL = {"bf16": 4e-3, "f16": 1e-3}


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


def dev_x(xbits, dtype):
    return torch.from_numpy(np.ascontiguousarray(xbits)).view(torch.float16 if dtype == "f16" else torch.bfloat16).cuda()


def _check(lqm, handle, p, fmt, xbits, xdt):
    w = lqm.QuantWeights.from_host(p, fmt)
    y = handle.gemm(w, dev_x(xbits, xdt))
    torch.cuda.synchronize()
    Weff = O.dequant_2bit(p) if fmt == lqm.FMT_2BIT else O.dequant_nf4(p)
    yref, E = O.matmul_ref(Weff, xbits, xdt)
    return assert_within(y.cpu().numpy(), yref, E, TOL[xdt], f"gemm fmt={fmt} x={xdt}")


@pytest.mark.parametrize("xdt", ["bf16", "f16"])
@pytest.mark.parametrize("shape", [(256, 128, 256), (300, 200, 1088), (1, 130, 512), (513, 384, 640)])
def test_gemm_2bit(lqm, handle, xdt, shape):
    M, N, K = shape
    p, outl = quantized_2bit(N, K, seed=M + N + K)
    xb = x_for(M, K, xdt, outl, seed=M)
    _check(lqm, handle, p, lqm.FMT_2BIT, xb, xdt)


@pytest.mark.parametrize("xdt", ["bf16", "f16"])
@pytest.mark.parametrize("shape", [(256, 128, 256), (300, 200, 1088), (17, 64, 128)])
def test_gemm_nf4(lqm, handle, xdt, shape):
    M, N, K = shape
    p = quantized_nf4(N, K, seed=M * 3 + K)
    xb = x_for(M, K, xdt, None, seed=M + 1)
    _check(lqm, handle, p, lqm.FMT_NF4, xb, xdt)


def test_gemm_no_anchors(lqm, handle):
    W = synth.weights(160, 512, 0.02, seed=9)
    p = O.quantize_2bit(W, np.zeros(0, np.int32))
    xb = x_for(260, 512, "bf16", None, seed=9)
    _check(lqm, handle, p, lqm.FMT_2BIT, xb, "bf16")


def test_gemm_agrees_with_gemv_on_small_m(lqm, handle):
    """Both entry points multiply the same weights: their outputs meet each other's bound."""
    N, K, M = 256, 1024, 8
    p, outl = quantized_2bit(N, K, seed=31)
    w = lqm.QuantWeights.from_host(p, lqm.FMT_2BIT)
    xb = x_for(M, K, "f16", outl, seed=31)
    x = dev_x(xb, "f16")
    y1 = handle.gemm(w, x).cpu().numpy().astype(np.float64)
    y2 = handle.gemv(w, x).cpu().numpy().astype(np.float64)
    _, E = O.matmul_ref(O.dequant_2bit(p), xb, "f16")
    assert np.all(np.abs(y1 - y2) <= 2e-3 * E + 1e-30)


@pytest.mark.parametrize("fmt", ["2bit", "nf4"])
def test_gemm_14b_layer_prefill_sampled(lqm, handle, fmt):
    """M = 2048 prefill over the 14B-layer down projection (5120 x 13824) and gate (13824 x 5120)."""
    g = np.random.default_rng(5)
    for i, (name, N, K) in enumerate([s for s in synth.LAYER_SHAPES["14b"] if s[0] in ("down", "gate")]):
        M = 2048
        outl = synth.outlier_channels(K, 0.01, seed=5)
        xb = synth.activations(M, K, "bf16", synth.channel_sigma(K, outl, 20.0), seed=5, matrix_id=i)
        if fmt == "2bit":
            pk = synth.random_packed_2bit(N, K, O.anchor_count(K), seed=5, matrix_id=i)
            w = lqm.QuantWeights.from_host(pk, lqm.FMT_2BIT)
        else:
            pk = synth.random_packed_nf4(N, K, seed=5, matrix_id=i)
            w = lqm.QuantWeights.from_host(pk, lqm.FMT_NF4)
        y = handle.gemm(w, dev_x(xb, "bf16")).cpu().numpy()
        rows = sorted(set(g.choice(N, 5, replace=False).tolist()) | {0, N - 1})
        for n in rows:
            if fmt == "2bit":
                yr = O.gemv_2bit_rows(pk, xb, "bf16", n, n + 1)
                one = {k: (v[n:n + 1] if k in ("codes", "scales", "offsets", "anchor_w") else v) for k, v in pk.items()}
                one["N"] = 1
                E = O.row_error_scale(O.dequant_2bit(one), xb, "bf16")
            else:
                yr = O.gemv_nf4_rows(pk, xb, "bf16", n, n + 1)
                E = O.row_error_scale(O.dequant_nf4(dict(codes=pk["codes"][n:n + 1], absmax=pk["absmax"][n:n + 1],
                                                         N=1, K=K)), xb, "bf16")
            assert_within(y[:, n:n + 1], yr, E, TOL["bf16"], f"{fmt} {name} row {n}")


@pytest.mark.parametrize("fmt", ["2bit", "nf4"])
def test_gemm_grouped_mixed_shapes(lqm, handle, fmt):
    """Problems of different N, K (and anchor counts) in one launch: each matches the oracle, and
    bit for bit its own lq_gemm call (every tile computes the same way on whichever CTA runs it)."""
    shapes = [(300, 200, 1088), (300, 384, 640), (300, 128, 256)]
    mats, probs = [], []
    for i, (M, N, K) in enumerate(shapes):
        if fmt == "2bit":
            p, outl = quantized_2bit(N, K, seed=40 + i)
            w = lqm.QuantWeights.from_host(p, lqm.FMT_2BIT)
            Weff = O.dequant_2bit(p)
        else:
            p, outl = quantized_nf4(N, K, seed=40 + i), None
            w = lqm.QuantWeights.from_host(p, lqm.FMT_NF4)
            Weff = O.dequant_nf4(p)
        xb = x_for(M, K, "bf16", outl, seed=40 + i)
        x = dev_x(xb, "bf16")
        y = torch.empty((M, N), dtype=torch.float32, device="cuda")
        mats.append((w, x, y, xb, Weff))
        probs.append(handle.problem(w, x, y))
    for _ in range(2):   # the second call reuses the resident schedule
        handle.gemm_grouped(probs)
        torch.cuda.synchronize()
        for (w, x, y, xb, Weff) in mats:
            yref, E = O.matmul_ref(Weff, xb, "bf16")
            assert_within(y.cpu().numpy(), yref, E, TOL["bf16"], f"grouped {fmt}")
            y1 = handle.gemm(w, x)
            assert torch.equal(y1, y)


# ---------------------------------------------------------------- 16-bit outputs

TDT = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


def gpu_bits(t):
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("ydt", ["bf16", "f16"])
@pytest.mark.parametrize("shape", [(300, 200, 1088), (256, 128, 256), (1, 130, 512), (513, 384, 640), (2048, 264, 512)])
def test_gemm_2bit_16bit_output(lqm, handle, ydt, shape):
    """16-bit y is the RNE rounding of the fp32 result, bit for bit, over ragged token tiles, row
    counts that are not a multiple of 8, and row tiles whose second CTA holds no rows."""
    M, N, K = shape
    p, outl = quantized_2bit(N, K, seed=M + N + K + 3)
    xb = x_for(M, K, "bf16", outl, seed=M + 3)
    w = lqm.QuantWeights.from_host(p, lqm.FMT_2BIT)
    x = dev_x(xb, "bf16")
    y16 = handle.gemm(w, x, y_dtype=TDT[ydt])
    y32 = handle.gemm(w, x)
    torch.cuda.synchronize()
    assert np.array_equal(gpu_bits(y16), O.round_to(y32.cpu().numpy(), ydt))


def test_gemm_grouped_mixed_output_dtypes(lqm, handle):
    """One grouped launch over problems with different output dtypes: each output equals its own
    single call bit for bit."""
    cases = [((300, 200, 1088), "bf16"), ((300, 130, 512), "bf16"), ((300, 384, 640), "f32"), ((300, 128, 256), "f16")]
    mats, probs = [], []
    for i, ((M, N, K), ydt) in enumerate(cases):
        p, outl = quantized_2bit(N, K, seed=50 + i)
        w = lqm.QuantWeights.from_host(p, lqm.FMT_2BIT)
        x = dev_x(x_for(M, K, "bf16", outl, seed=50 + i), "bf16")
        y = torch.empty((M, N), dtype=TDT[ydt], device="cuda")
        mats.append((w, x, y, ydt))
        probs.append(handle.problem(w, x, y))
    for _ in range(2):
        handle.gemm_grouped(probs)
        torch.cuda.synchronize()
        for (w, x, y, ydt) in mats:
            y1 = handle.gemm(w, x, y_dtype=TDT[ydt])
            assert torch.equal(y1, y)
