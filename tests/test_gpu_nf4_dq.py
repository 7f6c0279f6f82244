"""GPU parity of NF4 with double quantization (QLoRA's second quantization of the block
maxima, 8-bit floats in blocks of 256) against the CPU oracle, through the C ABI.

* lq_dequant: bit-exact, every element and output dtype;
* lq_gemv: |y - y_ref| <= 1e-3 * sum_k |W_eff||x| per output on the streaming kernel
  (K % 256 == 0) and the split-K kernel, 1..32 tokens, binary16 and bf16 x, batched, and a
  whole 7B decoder layer at full size on sampled rows;
* lq_gemm (the maxima decoded into the workspace, then the NF4 tcgen05 GEMM) within
  4e-3 * E (bf16 operands) or 1e-3 * E (fp16), single and grouped;
* the layer stream does not take this format.
"""
import numpy as np
import pytest

import synth
from oracle import oracle as O
from tests._util import assert_within, x_for

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

GEMV_TOL = 1e-3
TDT = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


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


def packed(N, K, seed):
    W = synth.weights(N, K, 0.02, seed=seed, big_frac=0.001, big_mult=10.0)
    return O.quantize_nf4_dq(W)


def dev_x(xbits, dtype):
    return torch.from_numpy(np.ascontiguousarray(xbits)).view(torch.float16 if dtype == "f16" else torch.bfloat16).cuda()


def gpu_bits(t):
    a = t.cpu()
    if a.dtype == torch.float32:
        return a.numpy().view(np.uint32)
    return a.view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("shape", [(512, 256), (130, 4096), (3, 64), (96, 1088)])
@pytest.mark.parametrize("odt", ["f32", "f16", "bf16"])
def test_dequant_nf4_dq_bit_exact(lqm, handle, shape, odt):
    N, K = shape
    p = packed(N, K, seed=N + K)
    w = lqm.QuantWeights.from_host(p, lqm.FMT_NF4_DQ)
    out = handle.dequant(w, out_dtype=TDT[odt])
    torch.cuda.synchronize()
    ref = O.round_to(O.dequant_nf4_dq(p), odt)
    assert np.array_equal(gpu_bits(out), ref.view(np.uint32) if odt == "f32" else ref)


def test_dequant_nf4_dq_every_maximum_code(lqm, handle):
    """Every finite 8-bit float code as a block maximum (both signs, subnormals, 448)."""
    N, K = 16, 1024                                  # 256 maxima = one second-level block
    codes = np.arange(256, dtype=np.uint8)
    codes[codes == 0x7F] = 0x7E
    codes[codes == 0xFF] = 0xFE
    p = dict(codes=np.full((N, K // 2), 0xE1, np.uint8), acodes=codes.reshape(N, K // 64),
             second=np.array([0.25, 1.0 / 448], np.float32), N=N, K=K)
    w = lqm.QuantWeights.from_host(p, lqm.FMT_NF4_DQ)
    out = handle.dequant(w, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert np.array_equal(gpu_bits(out), O.dequant_nf4_dq(p).view(np.uint32))


def _gemv(lqm, handle, p, xb, xdt):
    w = lqm.QuantWeights.from_host(p, lqm.FMT_NF4_DQ)
    y = handle.gemv(w, dev_x(xb, xdt), y_dtype=torch.float32)
    torch.cuda.synchronize()
    yref, E = O.matmul_ref(O.dequant_nf4_dq(p), xb, xdt)
    assert_within(y.cpu().numpy(), yref, E, GEMV_TOL, f"nf4-dq M={xb.shape[0]} K={p['K']}")
    handle.sync()


@pytest.mark.parametrize("M", [1, 4, 9, 16, 32])
@pytest.mark.parametrize("xdt", ["f16", "bf16"])
@pytest.mark.parametrize("K", [2048, 1088])
def test_gemv_nf4_dq_small(lqm, handle, M, xdt, K):
    # K = 2048: the streaming kernel; K = 1088 (not a multiple of 256): the split-K kernel
    N = 200
    p = packed(N, K, seed=M + K)
    _gemv(lqm, handle, p, x_for(M, K, xdt, seed=M), xdt)


@pytest.mark.parametrize("M", [1, 16])
def test_gemv_nf4_dq_split_k_forced(lqm, handle, monkeypatch, M):
    monkeypatch.setenv("LQ_GEMV_KERNEL", "regs")
    p = packed(130, 3072, seed=5 + M)
    _gemv(lqm, handle, p, x_for(M, 3072, "bf16", seed=5), "bf16")


def test_gemv_nf4_dq_batched(lqm, handle):
    L, N, K = 4, 48, 1024            # 768 maxima: 3 second-level blocks, 4 floats per member
    packs = [packed(N, K, seed=20 + l) for l in range(L)]
    st = lambda k: np.stack([p[k] for p in packs])
    big = dict(codes=st("codes"), acodes=st("acodes"), second=st("second"), N=N, K=K)
    w = lqm.QuantWeights.from_host(big, lqm.FMT_NF4_DQ)
    xs = np.stack([x_for(2, K, "bf16", seed=l) for l in range(L)])
    x = dev_x(xs, "bf16")
    y = torch.empty((L, 2, N), dtype=torch.float32, device="cuda")
    nsec = big["second"].shape[1]
    strides = dict(codes=N * K // 2, scales=N * K // 64, offsets=4 * nsec, x=2 * K * 2, y=2 * N * 4)
    if any(v % 16 for v in strides.values()):
        pytest.skip("member strides not 16-byte aligned for this shape")
    handle.gemv_grouped([handle.problem(w, x[0], y[0], batch=L, strides=strides)])
    torch.cuda.synchronize()
    for l in range(L):
        yref, E = O.matmul_ref(O.dequant_nf4_dq(packs[l]), xs[l], "bf16")
        assert_within(y[l].cpu().numpy(), yref, E, GEMV_TOL, f"member {l}")


@pytest.mark.parametrize("M", [1, 4])
def test_gemv_nf4_dq_7b_layer_sampled(lqm, handle, M):
    probs, keep = [], []
    for i, (name, N, K) in enumerate(synth.LAYER_SHAPES["7b"]):
        pk = synth.random_packed_nf4_dq(N, K, seed=6, matrix_id=i)
        w = lqm.QuantWeights.from_host(pk, lqm.FMT_NF4_DQ)
        xb = synth.activations(M, K, "bf16", None, seed=6, matrix_id=i)
        x = dev_x(xb, "bf16")
        y = torch.empty((M, N), dtype=torch.float32, device="cuda")
        probs.append(handle.problem(w, x, y))
        keep.append((pk, xb, y, w, x))
    handle.gemv_grouped(probs)
    torch.cuda.synchronize()
    for i, (pk, xb, y, _, _) in enumerate(keep):
        yc = y.cpu().numpy()
        g = np.random.default_rng(i)
        for n in sorted(set(g.choice(pk["N"], 3, replace=False).tolist()) | {pk["N"] - 1}):
            # rows 0..n keep the maxima's row-major indices (and so their second-level blocks)
            head = dict(pk, codes=pk["codes"][:n + 1], acodes=pk["acodes"][:n + 1], N=n + 1)
            Wn = O.dequant_nf4_dq(head)[n:n + 1]
            yref, E = O.matmul_ref(Wn, xb, "bf16")
            assert_within(yc[:, n:n + 1], yref, E, GEMV_TOL, f"7b[{i}] row {n}")


@pytest.mark.parametrize("xdt", ["bf16", "f16"])
@pytest.mark.parametrize("shape", [(256, 128, 256), (300, 200, 1088), (17, 64, 128)])
def test_gemm_nf4_dq(lqm, handle, xdt, shape):
    """Prefill: the maxima decoded into the workspace, then the tcgen05 NF4 GEMM (4e-3 * E
    with bf16 operands, 1e-3 * E with fp16)."""
    M, N, K = shape
    p = packed(N, K, seed=M + N + K)
    w = lqm.QuantWeights.from_host(p, lqm.FMT_NF4_DQ)
    xb = x_for(M, K, xdt, seed=M)
    y = handle.gemm(w, dev_x(xb, xdt), y_dtype=torch.float32)
    torch.cuda.synchronize()
    yref, E = O.matmul_ref(O.dequant_nf4_dq(p), xb, xdt)
    assert_within(y.cpu().numpy(), yref, E, 4e-3 if xdt == "bf16" else 1e-3, f"gemm nf4-dq {shape} {xdt}")
    handle.sync()


def test_gemm_nf4_dq_grouped(lqm, handle):
    shapes = [(256, 192, 512), (256, 64, 1024)]
    probs, keep = [], []
    for i, (M, N, K) in enumerate(shapes):
        p = packed(N, K, seed=70 + i)
        w = lqm.QuantWeights.from_host(p, lqm.FMT_NF4_DQ)
        xb = x_for(M, K, "bf16", seed=70 + i)
        x = dev_x(xb, "bf16")
        y = torch.empty((M, N), dtype=torch.float32, device="cuda")
        probs.append(handle.problem(w, x, y))
        keep.append((p, xb, y, w, x))
    handle.gemm_grouped(probs)
    torch.cuda.synchronize()
    for i, (p, xb, y, _, _) in enumerate(keep):
        yref, E = O.matmul_ref(O.dequant_nf4_dq(p), xb, "bf16")
        assert_within(y.cpu().numpy(), yref, E, 4e-3, f"grouped nf4-dq {i}")
    handle.sync()


def test_nf4_dq_layer_stream_refused(lqm, handle):
    """The layer stream carries 2-bit and NF4 layers only: a double-quantized layer is refused
    before any copy."""
    from bit_weight_quantized_dequant_gb300._lq import lq_problem
    N, K, M = 64, 256, 1
    p = lq_problem()
    p.format, p.M, p.N, p.K = lqm.FMT_NF4_DQ, M, N, K
    p.codes, p.scales, p.offsets = 0, 1024, 2048            # byte offsets into the layer blob
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    x = torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
    p.x, p.x_dtype, p.y, p.y_dtype, p.batch = x.data_ptr(), lqm.BF16, y.data_ptr(), lqm.F32, 1
    host = torch.zeros(4096, dtype=torch.uint8).pin_memory()
    s = lqm.LayerStream(handle, 1 << 20)
    try:
        with pytest.raises(lqm.LQError) as e:
            s.run(host, 4096, 4096, 1, [p])
        assert e.value.status == lqm.LQ_ERR_UNSUPPORTED
    finally:
        s.close()
    handle.sync()
