"""lq_gemv_noalloc: the decode product for callers that may not allocate device memory.

Such callers (a plugin inside an application that owns all device memory, or a
service that must not allocate after start-up) cannot create a handle, because
lq_create allocates the handle's workspace.  lq_gemv_noalloc takes no handle and
keeps its scratch in a fixed device array inside the library.  These tests call it
through the C ABI on each decode kernel it can reach (the ring kernel at 4 tokens and
K % 256 == 0, the streaming kernel at 12 tokens, the split-K kernel when K % 256 != 0)
and compare every output with the oracle's y_ref, within the GEMV bound
(1e-3 * sum_k |W_eff||x|), on two calls in a row.  The file name keeps it last in
collection order, so a run that stops at the first failure has already run every
other test.
"""
import ctypes

import numpy as np
import pytest

from oracle import oracle as O
import synth
from tests._util import quantized_2bit, quantized_int4, x_for

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

TOL = 1e-3


@pytest.fixture(scope="module")
def lqm():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import bit_weight_quantized_dequant_gb300 as lq
    lq.build()
    return lq


def _noalloc(L, w, x, y, stream=None):
    fmt, c, s, o, ai, aw, A, ld = w.args()
    xdt = 2 if x.dtype == torch.bfloat16 else 1
    return L.lq_gemv_noalloc(fmt, c, s, o, ai, aw, A, ld, x.data_ptr(), xdt, y.data_ptr(), 0, x.shape[0], w.N, w.K,
                             stream)


@pytest.mark.parametrize("N,K,M", [(700, 11008, 4), (700, 11008, 12), (700, 11040, 4)])
def test_noalloc_matches_the_oracle_on_two_calls_in_a_row(lqm, N, K, M):
    torch.cuda.set_device(0)
    L = lqm.load_library()
    # K = 11040 is not a multiple of 256: the split-K kernel, whose partial sums (6 K-parts
    # plus an anchor part per 64-row strip) live in the scratch; the other two use it for
    # row-block slots
    p, outl = quantized_2bit(N, K, seed=77 + M)
    w = lqm.QuantWeights.from_host(p, lqm.FMT_2BIT)
    xb = x_for(M, K, "f16", outl, seed=77)
    x = torch.from_numpy(xb).view(torch.float16).cuda()
    y_ref, E = O.matmul_ref(O.dequant_2bit(p), xb, "f16")
    for call in range(2):
        y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        st = _noalloc(L, w, x, y)
        assert st == lqm.LQ_OK, L.lq_status_string(st)
        torch.cuda.synchronize()
        got = y.cpu().numpy().astype(np.float64)
        assert np.all(np.isfinite(got)), f"call {call}: unwritten outputs"
        err = np.abs(got - y_ref)
        assert np.all(err <= TOL * E + 1e-30), f"call {call}: max err/E = {np.max(err / (E + 1e-30)):.3e}"


@pytest.mark.parametrize("fmt", ["int4", "nf4_dq"])
def test_noalloc_other_formats_match_the_oracle(lqm, fmt):
    """INT4 (the ring kernel, x gathered through the permutation) and NF4 with double
    quantization (the streaming kernel) through the same entry point."""
    L = lqm.load_library()
    N, K, M = 700, 4096, 4
    if fmt == "int4":
        p, outl = quantized_int4(N, K, seed=5)
        w = lqm.QuantWeights.from_host(p, lqm.FMT_INT4)
        W = O.dequant_int4(p)
    else:
        p = O.quantize_nf4_dq(synth.weights(N, K, 0.02, seed=6, big_frac=0.001, big_mult=10.0))
        outl = None
        w = lqm.QuantWeights.from_host(p, lqm.FMT_NF4_DQ)
        W = O.dequant_nf4_dq(p)
    xb = x_for(M, K, "bf16", outl, seed=7)
    x = torch.from_numpy(xb).view(torch.bfloat16).cuda()
    y_ref, E = O.matmul_ref(W, xb, "bf16")
    for call in range(2):
        y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        st = _noalloc(L, w, x, y)
        assert st == lqm.LQ_OK, L.lq_status_string(st)
        torch.cuda.synchronize()
        err = np.abs(y.cpu().numpy().astype(np.float64) - y_ref)
        assert np.all(err <= TOL * E + 1e-30), f"{fmt} call {call}: max err/E = {np.max(err / (E + 1e-30)):.3e}"


def test_noalloc_rejects_problems_beyond_its_scratch(lqm):
    L = lqm.load_library()
    # K % 256 != 0 takes the split-K kernel, whose partial sums here (~4.5 M floats) exceed the scratch
    N, K, M = 8192, 8224, 32
    codes = torch.zeros((N, K // 4), dtype=torch.uint8, device="cuda")
    sc = torch.zeros((N, K // 32), dtype=torch.float16, device="cuda")
    x = torch.zeros((M, K), dtype=torch.float16, device="cuda")
    y = torch.full((M, N), 3.0, dtype=torch.float32, device="cuda")
    st = L.lq_gemv_noalloc(1, codes.data_ptr(), sc.data_ptr(), sc.data_ptr(), None, None, 0, 0, x.data_ptr(), 1,
                           y.data_ptr(), 0, M, N, K, None)
    assert st == lqm.LQ_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.all(y == 3.0)
