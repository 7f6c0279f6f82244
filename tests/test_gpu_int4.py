"""GPU parity of the INT4 format (otf-llm README, the v3.2 engine) against the CPU oracle.

* lq_dequant: bit-exact for every element and output dtype (S * q is exact in fp32, and
  each value lands at its input column perm[j]; anchor columns carry their binary16 value);
* lq_gemv (the ring kernel, K % 256 == 0): |y - y_ref| <= 1e-3 * sum_k |W_eff||x| per
  output, for 1..32 tokens, binary16 and bf16 x, ragged row counts, x built in shared
  memory and by the pre-pass, grouped and batched problems, a whole 7B decoder layer at
  full size on sampled rows, bf16 x far outside binary16's range, and the weight range
  limit (8 |S| >= 65520 reports LQ_ERR_RANGE);
* lq_gemm (prefill on tcgen05): 4e-3 * E (bf16) / 1e-3 * E (fp16), single and grouped;
* a decode with K % 256 != 0 answers LQ_ERR_UNSUPPORTED without launching.
"""
import numpy as np
import pytest

import synth
from oracle import oracle as O
from tests._util import assert_within, quantized_int4, x_for

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


def dev_x(xbits, dtype):
    t = torch.from_numpy(np.ascontiguousarray(xbits)).view(torch.float16 if dtype == "f16" else torch.bfloat16)
    return t.cuda()


def gpu_bits(t):
    a = t.cpu()
    if a.dtype == torch.float32:
        return a.numpy().view(np.uint32)
    return a.view(torch.int16).numpy().view(np.uint16)


def gemv_check(lqm, handle, p, xbits, xdt, what=""):
    w = lqm.QuantWeights.from_host(p, lqm.FMT_INT4)
    y = handle.gemv(w, dev_x(xbits, xdt), y_dtype=torch.float32)
    torch.cuda.synchronize()
    yref, E = O.matmul_ref(O.dequant_int4(p), xbits, xdt)
    r = assert_within(y.cpu().numpy(), yref, E, GEMV_TOL, f"int4 {what} M={xbits.shape[0]}")
    handle.sync()
    return r


# ---------------------------------------------------------------- dequant

@pytest.mark.parametrize("shape", [(512, 256), (200, 2592), (7, 32), (65, 4096)])
@pytest.mark.parametrize("odt", ["f32", "f16", "bf16"])
def test_dequant_int4_bit_exact(lqm, handle, shape, odt):
    N, K = shape
    p, _ = quantized_int4(N, K, seed=N + 3 * K)
    w = lqm.QuantWeights.from_host(p, lqm.FMT_INT4)
    out = handle.dequant(w, out_dtype=TDT[odt])
    torch.cuda.synchronize()
    ref = O.round_to(O.dequant_int4(p), odt)
    got = gpu_bits(out)
    assert np.array_equal(got, ref.view(np.uint32) if odt == "f32" else ref)


def test_dequant_int4_every_code_at_every_position(lqm, handle):
    """All 16 codes (-8..7, -8 included although the quantizer never writes it) at every
    nibble position, a non-trivial permutation, no anchors."""
    N, K = 16, 256
    q = ((np.arange(N)[:, None] + np.arange(K)[None, :]) % 16 - 8).astype(np.int8)
    g = np.random.default_rng(5)
    S = (g.uniform(0.5, 2.0, size=(N, K // 32)) * 1e-2).astype(np.float16)
    p = dict(codes=O.pack_int4(q), scales=S.view(np.uint16), perm=g.permutation(K).astype(np.int32),
             anchor_idx=np.zeros(0, np.int32), anchor_w=np.zeros((N, 8), np.uint16), A=0, ld_anchor=8, N=N, K=K)
    w = lqm.QuantWeights.from_host(p, lqm.FMT_INT4)
    out = handle.dequant(w, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert np.array_equal(gpu_bits(out), O.dequant_int4(p).view(np.uint32))
    # and the same codes through the GEMV
    xb = x_for(3, K, "f16", seed=5)
    gemv_check(lqm, handle, p, xb, "f16", "all codes")


# ---------------------------------------------------------------- gemv, small shapes (every output)

@pytest.mark.parametrize("M", [1, 2, 4, 7, 8, 9, 16, 24, 32])
@pytest.mark.parametrize("xdt", ["f16", "bf16"])
def test_gemv_int4_small(lqm, handle, M, xdt):
    # 200 rows = 6 full 32-row units and a ragged one; K = 2560 = 10 steps of 256
    N, K = 200, 2560
    p, outl = quantized_int4(N, K, seed=7)
    xb = x_for(M, K, xdt, outl, seed=7 + M)
    gemv_check(lqm, handle, p, xb, xdt)


@pytest.mark.parametrize("M", [1, 4, 16])
def test_gemv_int4_x_from_the_pre_pass(lqm, handle, monkeypatch, M):
    """LQ_GEMV_XS=0: x gathered through the permutation by the pre-pass into global memory
    instead of by each CTA into shared memory."""
    monkeypatch.setenv("LQ_GEMV_XS", "0")
    for xdt in ("f16", "bf16"):
        p, outl = quantized_int4(300, 3072, seed=9 + M)
        xb = x_for(M, 3072, xdt, outl, seed=9 + M)
        gemv_check(lqm, handle, p, xb, xdt, "pre-pass")


@pytest.mark.parametrize("shape", [(512, 256), (33, 256), (1, 4096), (96, 8192)])
def test_gemv_int4_shapes(lqm, handle, shape):
    N, K = shape
    p, outl = quantized_int4(N, K, seed=N + 11)
    xb = x_for(1, K, "f16", outl, seed=N)
    gemv_check(lqm, handle, p, xb, "f16", f"{N}x{K}")


def test_gemv_int4_no_anchors_identity_perm(lqm, handle):
    N, K = 64, 512
    W = synth.weights(N, K, 0.02, seed=2)
    p = O.quantize_int4(W, np.arange(K, dtype=np.int32), np.zeros(0, np.int32))
    gemv_check(lqm, handle, p, x_for(4, K, "f16", seed=2), "f16", "no anchors")


def test_gemv_int4_grouped_and_batched(lqm, handle):
    """Four problems of different shapes in one call, then one problem of five members with
    distinct weights, permutations and x (member strides in bytes)."""
    shapes = [(96, 512), (96, 512), (200, 768), (40, 1024)]
    probs, keep = [], []
    for i, (N, K) in enumerate(shapes):
        p, outl = quantized_int4(N, K, seed=40 + i)
        w = lqm.QuantWeights.from_host(p, lqm.FMT_INT4)
        xb = x_for(3, K, "f16", outl, seed=40 + i)
        x = dev_x(xb, "f16")
        y = torch.empty((3, N), dtype=torch.float32, device="cuda")
        probs.append(handle.problem(w, x, y))
        keep.append((p, xb, y, w, x))
    handle.gemv_grouped(probs)
    torch.cuda.synchronize()
    for i, (p, xb, y, _, _) in enumerate(keep):
        yref, E = O.matmul_ref(O.dequant_int4(p), xb, "f16")
        assert_within(y.cpu().numpy(), yref, E, GEMV_TOL, f"grouped {i}")

    L, N, K = 5, 128, 1024
    packs = [synth.random_packed_int4(N, K, 8, seed=l) for l in range(L)]
    st = lambda key: np.stack([p[key] for p in packs])
    big = dict(codes=st("codes"), scales=st("scales"), perm=st("perm"), anchor_idx=st("anchor_idx"),
               anchor_w=st("anchor_w"), A=8, ld_anchor=packs[0]["ld_anchor"], N=N, K=K)
    w = lqm.QuantWeights.from_host(big, lqm.FMT_INT4)
    xs = np.stack([synth.activations(2, K, "bf16", seed=l) for l in range(L)])
    x = dev_x(xs, "bf16")
    y = torch.empty((L, 2, N), dtype=torch.float32, device="cuda")
    strides = dict(codes=N * K // 2, scales=N * K // 32 * 2, offsets=4 * K, anchor_idx=4 * 8,
                   anchor_w=N * big["ld_anchor"] * 2, x=2 * K * 2, y=2 * N * 4)
    handle.gemv_grouped([handle.problem(w, x[0], y[0], batch=L, strides=strides)])
    torch.cuda.synchronize()
    for l in range(L):
        yref, E = O.matmul_ref(O.dequant_int4(packs[l]), xs[l], "bf16")
        assert_within(y[l].cpu().numpy(), yref, E, GEMV_TOL, f"batch member {l}")


# ---------------------------------------------------------------- full size, sampled rows

@pytest.mark.parametrize("M", [1, 4, 16])
def test_gemv_int4_7b_layer_sampled(lqm, handle, M):
    """A whole 7B decoder layer (7 projections, 1% binary16 columns) in one grouped call."""
    probs, keep = [], []
    for i, (name, N, K) in enumerate(synth.LAYER_SHAPES["7b"]):
        pk = synth.random_packed_int4(N, K, int(np.floor(O.INT4_OUTLIER_FRAC * K)), seed=4, matrix_id=i)
        w = lqm.QuantWeights.from_host(pk, lqm.FMT_INT4)
        xb = synth.activations(M, K, "bf16", synth.channel_sigma(K, synth.outlier_channels(K, 0.01, seed=4)),
                               seed=4, matrix_id=i)
        x = dev_x(xb, "bf16")
        y = torch.empty((M, N), dtype=torch.float32, device="cuda")
        probs.append(handle.problem(w, x, y))
        keep.append((pk, xb, y, w, x))
    handle.gemv_grouped(probs)
    torch.cuda.synchronize()
    for i, (pk, xb, y, _, _) in enumerate(keep):
        yc = y.cpu().numpy()
        g = np.random.default_rng(i)
        for n in sorted(set(g.choice(pk["N"], 6, replace=False).tolist()) | {0, pk["N"] - 1}):
            one = dict(pk, codes=pk["codes"][n:n + 1], scales=pk["scales"][n:n + 1],
                       anchor_w=pk["anchor_w"][n:n + 1], N=1)
            yref, E = O.matmul_ref(O.dequant_int4(one), xb, "bf16")
            assert_within(yc[:, n:n + 1], yref, E, GEMV_TOL, f"7b[{i}] row {n}")


# ---------------------------------------------------------------- operand domain

@pytest.mark.parametrize("M", [1, 5, 12])
@pytest.mark.parametrize("mag", [1e5, 1e-6, "mixed"])
def test_gemv_int4_bf16_x_magnitudes(lqm, handle, M, mag):
    N, K = 150, 2048
    p, outl = quantized_int4(N, K, seed=M + 21)
    scales = np.array([1e5 if (mag == 1e5 or (mag == "mixed" and m % 2 == 0)) else 1e-6 for m in range(M)])
    base = O.x_values(x_for(M, K, "bf16", outl, seed=M), "bf16")
    xb = O.round_to((base * scales[:, None]).astype(np.float32), "bf16")
    gemv_check(lqm, handle, p, xb, "bf16", f"mag={mag}")


def test_gemv_int4_weight_range_limit(lqm, handle):
    """A group scale of 8000 (|S q| <= 64000) stays inside binary16 and meets the bound; 9000
    (8 * 9000 = 72000) is accepted and the next lq_sync reports LQ_ERR_RANGE."""
    N, K, M = 96, 1024, 2
    p, outl = quantized_int4(N, K, seed=31)
    xb = x_for(M, K, "f16", outl, seed=31)
    for S, ok in ((8000.0, True), (9000.0, False)):
        q = dict(p, scales=p["scales"].copy())
        q["scales"][17, 5] = np.float16(S).view(np.uint16)
        if ok:
            gemv_check(lqm, handle, q, xb, "f16", "inside the range")
        else:
            w = lqm.QuantWeights.from_host(q, lqm.FMT_INT4)
            handle.gemv(w, dev_x(xb, "f16"))
            with pytest.raises(lqm.LQError) as e:
                handle.sync()
            assert e.value.status == lqm.LQ_ERR_RANGE
    gemv_check(lqm, handle, p, xb, "f16", "after the range error")


# ---------------------------------------------------------------- prefill (tcgen05 GEMM)

@pytest.mark.parametrize("xdt", ["bf16", "f16"])
@pytest.mark.parametrize("shape", [(256, 128, 256), (300, 200, 1088), (17, 64, 128), (513, 384, 640)])
def test_gemm_int4(lqm, handle, xdt, shape):
    """x permuted once into the workspace, two 16-entry S*q tables per 64-column block in the
    producer warps, the outlier columns as extra K-blocks: 4e-3 * E with bf16 operands, 1e-3 * E
    with fp16 (the weights are rounded once to the operand type)."""
    M, N, K = shape
    p, outl = quantized_int4(N, K, seed=M + N + K)
    w = lqm.QuantWeights.from_host(p, lqm.FMT_INT4)
    xb = x_for(M, K, xdt, outl, seed=M)
    y = handle.gemm(w, dev_x(xb, xdt), y_dtype=torch.float32)
    torch.cuda.synchronize()
    yref, E = O.matmul_ref(O.dequant_int4(p), xb, xdt)
    assert_within(y.cpu().numpy(), yref, E, 4e-3 if xdt == "bf16" else 1e-3, f"gemm int4 {shape} {xdt}")
    handle.sync()


def test_gemm_int4_grouped_and_all_codes(lqm, handle):
    """Two problems in one launch; the second holds every nibble (-8 included) at every position."""
    probs, keep = [], []
    p0, outl = quantized_int4(192, 512, seed=90)
    N, K = 64, 256
    q = ((np.arange(N)[:, None] + np.arange(K)[None, :]) % 16 - 8).astype(np.int8)
    g = np.random.default_rng(9)
    p1 = dict(codes=O.pack_int4(q), scales=(g.uniform(0.5, 2.0, size=(N, K // 32)) * 1e-2).astype(np.float16).view(np.uint16),
              perm=g.permutation(K).astype(np.int32), anchor_idx=np.zeros(0, np.int32), anchor_w=np.zeros((N, 8), np.uint16),
              A=0, ld_anchor=8, N=N, K=K)
    for i, p in enumerate((p0, p1)):
        w = lqm.QuantWeights.from_host(p, lqm.FMT_INT4)
        xb = x_for(256, p["K"], "bf16", outl if i == 0 else None, seed=91 + i)
        x = dev_x(xb, "bf16")
        y = torch.empty((256, p["N"]), dtype=torch.float32, device="cuda")
        probs.append(handle.problem(w, x, y))
        keep.append((p, xb, y, w, x))
    handle.gemm_grouped(probs)
    torch.cuda.synchronize()
    for i, (p, xb, y, _, _) in enumerate(keep):
        yref, E = O.matmul_ref(O.dequant_int4(p), xb, "bf16")
        assert_within(y.cpu().numpy(), yref, E, 4e-3, f"grouped int4 {i}")
    handle.sync()


def test_gemm_int4_14b_prefill_sampled(lqm, handle):
    """M = 2048 prefill over the 14B layer's down projection (5120 x 13824) and gate (13824 x 5120),
    sampled rows against the oracle."""
    g = np.random.default_rng(8)
    for i, (name, N, K) in enumerate([s for s in synth.LAYER_SHAPES["14b"] if s[0] in ("down", "gate")]):
        M = 2048
        outl = synth.outlier_channels(K, 0.01, seed=8)
        xb = synth.activations(M, K, "bf16", synth.channel_sigma(K, outl, 20.0), seed=8, matrix_id=i)
        pk = synth.random_packed_int4(N, K, int(np.floor(O.INT4_OUTLIER_FRAC * K)), seed=8, matrix_id=i)
        w = lqm.QuantWeights.from_host(pk, lqm.FMT_INT4)
        y = handle.gemm(w, dev_x(xb, "bf16")).float().cpu().numpy()
        for n in sorted(set(g.choice(N, 4, replace=False).tolist()) | {0, N - 1}):
            one = dict(pk, codes=pk["codes"][n:n + 1], scales=pk["scales"][n:n + 1], anchor_w=pk["anchor_w"][n:n + 1], N=1)
            yref, E = O.matmul_ref(O.dequant_int4(one), xb, "bf16")
            assert_within(y[:, n:n + 1], yref, E, 4e-3, f"int4 {name} row {n}")
    handle.sync()


# ---------------------------------------------------------------- what INT4 does not take

def test_int4_unsupported_paths_launch_nothing(lqm, handle):
    p, outl = quantized_int4(64, 2592, seed=1)             # K % 256 != 0: no decode kernel takes it
    w = lqm.QuantWeights.from_host(p, lqm.FMT_INT4)
    y = torch.full((1, 64), 7.0, device="cuda")
    x = dev_x(x_for(1, 2592, "f16", outl), "f16")
    with pytest.raises(lqm.LQError) as e:
        handle.gemv(w, x, y=y)
    assert e.value.status == lqm.LQ_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert torch.all(y == 7.0)
    handle.sync()
