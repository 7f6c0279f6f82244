"""The decode GEMV across the binary16 operand range of its tensor cores (GPU, through the C ABI).

* bf16 x far outside binary16's normal range (about 1e5 and about 1e-6, and both in one
  call on different tokens): each token is scaled by a power of two before the binary16
  rounding and back after the product, so the 1e-3 * sum|W_eff||x| bound still holds;
* 2-bit weights whose table values fmaf(S, C[q], Z) pass binary16's largest finite value:
  the call is accepted and the next lq_sync reports LQ_ERR_RANGE; values just inside the
  range meet the bound;
* every decode kernel: the ring kernel (2-bit, up to 8 tokens, K % 256 == 0), the
  streaming kernel (more tokens, and NF4) and the split-K kernel (K % 256 != 0).
"""
import numpy as np
import pytest

from oracle import oracle as O
from tests._util import assert_within, quantized_2bit, quantized_nf4, x_for

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

GEMV_TOL = 1e-3


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


def bf16_bits(v: np.ndarray) -> np.ndarray:
    """float64 values -> bf16 bit patterns, round to nearest even (via the oracle's C rounding)."""
    return O.round_to(np.asarray(v, dtype=np.float32), "bf16")


def scaled_bf16_x(M, K, scales, outl, seed):
    """bf16 x whose token m is N(0,1) (1% channels x20) times scales[m]."""
    base = O.x_values(x_for(M, K, "bf16", outl, seed=seed), "bf16")
    return bf16_bits(base * np.asarray(scales, dtype=np.float64)[:, None])


def run_gemv(lqm, handle, p, fmt, xbits, xdt="bf16"):
    w = lqm.QuantWeights.from_host(p, fmt)
    x = torch.from_numpy(np.ascontiguousarray(xbits)).view(torch.bfloat16 if xdt == "bf16" else torch.float16).cuda()
    y = handle.gemv(w, x, y_dtype=torch.float32)
    torch.cuda.synchronize()
    return y.cpu().numpy()


CASES = [  # (kernel forced, M, K): ring (M <= 8), streaming (M > 8), split-K (K % 256 != 0)
    ("ring", 1, 2048), ("ring", 5, 1536), ("stream", 12, 2048), ("regs", 3, 1056),
]


@pytest.mark.parametrize("kernel,M,K", CASES)
@pytest.mark.parametrize("mag", [1e5, 1e-6, "mixed"])
def test_bf16_x_magnitudes_2bit(lqm, handle, monkeypatch, kernel, M, K, mag):
    monkeypatch.setenv("LQ_GEMV_KERNEL", kernel)
    N = 150
    p, outl = quantized_2bit(N, K, seed=M + K)
    scales = [1e5 if (mag == 1e5 or (mag == "mixed" and m % 2 == 0)) else 1e-6 for m in range(M)]
    xb = scaled_bf16_x(M, K, scales, outl, seed=K + M)
    y = run_gemv(lqm, handle, p, lqm.FMT_2BIT, xb)
    yref, E = O.matmul_ref(O.dequant_2bit(p), xb, "bf16")
    assert_within(y, yref, E, GEMV_TOL, f"2-bit {kernel} M={M} mag={mag}")
    handle.sync()


@pytest.mark.parametrize("M", [1, 16])
@pytest.mark.parametrize("mag", [1e5, 1e-6, "mixed"])
def test_bf16_x_magnitudes_nf4(lqm, handle, M, mag):
    N, K = 130, 2048
    p = quantized_nf4(N, K, seed=M + 7)
    scales = [1e5 if (mag == 1e5 or (mag == "mixed" and m % 2 == 0)) else 1e-6 for m in range(M)]
    xb = scaled_bf16_x(M, K, scales, None, seed=M + 9)
    y = run_gemv(lqm, handle, p, lqm.FMT_NF4, xb)
    yref, E = O.matmul_ref(O.dequant_nf4(p), xb, "bf16")
    assert_within(y, yref, E, GEMV_TOL, f"nf4 M={M} mag={mag}")


def with_big_group(p, n, g, S, Z=0.0):
    """A copy of a 2-bit pack with row n, group g's scale and offset set to binary16(S), binary16(Z)."""
    q = dict(p)
    q["scales"] = p["scales"].copy()
    q["offsets"] = p["offsets"].copy()
    q["scales"][n, g] = np.float16(S).view(np.uint16)
    q["offsets"][n, g] = np.float16(Z).view(np.uint16)
    return q


@pytest.mark.parametrize("kernel,M,K", CASES)
def test_weight_range_limit(lqm, handle, monkeypatch, kernel, M, K):
    """|S*C+Z| reaches 65520 (1.52 * 50000): LQ_ERR_RANGE at the next lq_sync, and the handle
    keeps working; 1.52 * 40000 = 60800 stays inside and meets the bound."""
    monkeypatch.setenv("LQ_GEMV_KERNEL", kernel)
    N = 96
    p, outl = quantized_2bit(N, K, seed=3 * K + M)
    xb = x_for(M, K, "f16", outl, seed=K)
    g = 5 if 5 * 32 not in set(p["anchor_idx"].tolist()) else 6
    inside = with_big_group(p, 17, g, 40000.0)
    y = run_gemv(lqm, handle, inside, lqm.FMT_2BIT, xb, "f16")
    yref, E = O.matmul_ref(O.dequant_2bit(inside), xb, "f16")
    assert_within(y, yref, E, GEMV_TOL, f"{kernel} inside the range")
    handle.sync()
    outside = with_big_group(p, 17, g, 50000.0)
    run_gemv(lqm, handle, outside, lqm.FMT_2BIT, xb, "f16")
    with pytest.raises(lqm.LQError) as e:
        handle.sync()
    assert e.value.status == lqm.LQ_ERR_RANGE
    handle.sync()                       # the status was cleared
    y = run_gemv(lqm, handle, p, lqm.FMT_2BIT, xb, "f16")
    yref, E = O.matmul_ref(O.dequant_2bit(p), xb, "f16")
    assert_within(y, yref, E, GEMV_TOL, f"{kernel} after the range error")
    handle.sync()
