"""GPU parity of lq_dequant and lq_gemv against the CPU oracle (through the C ABI).

* dequant: bit-exact, every element, every format and output dtype;
* gemv: |y - y_ref| <= 1e-3 * sum_k |W_eff||x| per output (fp32 accumulation),
  on shapes that span several 64-row strips, several K splits and ragged tails,
  and at the full workload sizes on sampled rows.
"""
import numpy as np
import pytest

import synth
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


def dev_x(xbits, dtype):
    t = torch.from_numpy(np.ascontiguousarray(xbits)).view(torch.float16 if dtype == "f16" else torch.bfloat16)
    return t.cuda()


TDT = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


def gpu_bits(t):
    a = t.cpu()
    if a.dtype == torch.float32:
        return a.numpy()
    return a.view(torch.int16).numpy().view(np.uint16)


# ---------------------------------------------------------------- dequant

@pytest.mark.parametrize("shape", [(512, 256), (200, 2592), (7, 32), (65, 4096)])
@pytest.mark.parametrize("odt", ["f32", "f16", "bf16"])
def test_dequant_2bit_bit_exact(lqm, handle, shape, odt):
    N, K = shape
    p, _ = quantized_2bit(N, K, seed=N + K)
    w = lqm.QuantWeights.from_host(p, lqm.FMT_2BIT)
    out = handle.dequant(w, out_dtype=TDT[odt])
    torch.cuda.synchronize()
    ref = O.round_to(O.dequant_2bit(p), odt)
    got = gpu_bits(out)
    assert np.array_equal(got.view(np.uint32) if odt == "f32" else got,
                          ref.view(np.uint32) if odt == "f32" else ref)


@pytest.mark.parametrize("shape", [(512, 256), (130, 4096), (3, 64)])
@pytest.mark.parametrize("odt", ["f32", "f16", "bf16"])
def test_dequant_nf4_bit_exact(lqm, handle, shape, odt):
    N, K = shape
    p = quantized_nf4(N, K, seed=N * 7 + K)
    w = lqm.QuantWeights.from_host(p, lqm.FMT_NF4)
    out = handle.dequant(w, out_dtype=TDT[odt])
    torch.cuda.synchronize()
    ref = O.round_to(O.dequant_nf4(p), odt)
    got = gpu_bits(out)
    assert np.array_equal(got.view(np.uint32) if odt == "f32" else got,
                          ref.view(np.uint32) if odt == "f32" else ref)


def test_dequant_nf4_all_sixteen_levels(lqm, handle):
    """Every code in every position: the kernel's table equals the oracle's, bit for bit."""
    q = np.tile(np.arange(16, dtype=np.uint8), (4, 8))          # [4][128]
    p = dict(codes=O.pack_nf4(q), absmax=np.array([[1.0, 0.5], [2.0, 3.0], [0.1, 7.0], [1e-3, 0.0]], np.float32),
             N=4, K=128)
    w = lqm.QuantWeights.from_host(p, lqm.FMT_NF4)
    out = handle.dequant(w, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy().view(np.uint32), O.dequant_nf4(p).view(np.uint32))


# ---------------------------------------------------------------- gemv, small shapes (full oracle)

def _gemv_check(lqm, handle, p, fmt, xbits, xdt, ydt="f32", tol=GEMV_TOL):
    w = lqm.QuantWeights.from_host(p, fmt)
    x = dev_x(xbits, xdt)
    y = handle.gemv(w, x, y_dtype=TDT[ydt])
    torch.cuda.synchronize()
    Weff = O.dequant_2bit(p) if fmt == lqm.FMT_2BIT else O.dequant_nf4(p)
    yref, E = O.matmul_ref(Weff, xbits, xdt)
    return assert_within(y.float().cpu().numpy(), yref, E, tol, f"gemv fmt={fmt} M={xbits.shape[0]}")


@pytest.mark.parametrize("M", [1, 2, 4, 7, 8, 9, 16, 24, 32])
def test_gemv_2bit_small(lqm, handle, M):
    # 200 rows = 3 full strips + a ragged one; K = 2592 = 10 steps + 32 columns (ragged, non-16B rows)
    N, K = 200, 2592
    p, outl = quantized_2bit(N, K, seed=3)
    xb = x_for(M, K, "f16", outl, seed=3 + M)
    _gemv_check(lqm, handle, p, lqm.FMT_2BIT, xb, "f16")


@pytest.mark.parametrize("shape", [(512, 256), (64, 32), (1, 4096), (333, 1024), (96, 8192)])
def test_gemv_2bit_shapes(lqm, handle, shape):
    N, K = shape
    p, outl = quantized_2bit(N, K, seed=N + 5)
    xb = x_for(1, K, "f16", outl, seed=N)
    _gemv_check(lqm, handle, p, lqm.FMT_2BIT, xb, "f16")


def test_gemv_512x256_single_linear_workload(lqm, handle):
    """K=256, N=512, M=1, sigma 0.02, 8 anchors, seed 0."""
    W = synth.weights(512, 256, 0.02, seed=0, cfg=1)
    ai = O.select_anchors(W, O.activation_profile(np.ones(256)))
    assert len(ai) == 8
    p = O.quantize_2bit(W, ai)
    xb = synth.activations(1, 256, "f16", seed=0, cfg=1)
    _gemv_check(lqm, handle, p, lqm.FMT_2BIT, xb, "f16")


@pytest.mark.parametrize("ydt", ["f16", "bf16"])
def test_gemv_output_dtypes(lqm, handle, ydt):
    N, K = 150, 1024
    p, outl = quantized_2bit(N, K, seed=11)
    xb = x_for(3, K, "f16", outl, seed=11)
    w = lqm.QuantWeights.from_host(p, lqm.FMT_2BIT)
    y = handle.gemv(w, dev_x(xb, "f16"), y_dtype=TDT[ydt])
    y32 = handle.gemv(w, dev_x(xb, "f16"), y_dtype=torch.float32)
    torch.cuda.synchronize()
    # the narrow output is the RNE rounding of the fp32 result
    assert np.array_equal(gpu_bits(y), O.round_to(y32.cpu().numpy(), ydt))


@pytest.mark.parametrize("M", [1, 4, 16])
def test_gemv_nf4_small(lqm, handle, M):
    N, K = 130, 2560
    p = quantized_nf4(N, K, seed=M)
    xb = x_for(M, K, "bf16", None, seed=M)
    _gemv_check(lqm, handle, p, lqm.FMT_NF4, xb, "bf16")


def test_gemv_bf16_x_2bit(lqm, handle):
    N, K = 128, 1536
    p, outl = quantized_2bit(N, K, seed=21)
    xb = x_for(5, K, "bf16", outl, seed=21)
    _gemv_check(lqm, handle, p, lqm.FMT_2BIT, xb, "bf16")


def test_gemv_no_anchors_and_all_anchor_group(lqm, handle):
    W = synth.weights(70, 320, 0.02, seed=4)
    p0 = O.quantize_2bit(W, np.zeros(0, np.int32))
    xb = x_for(2, 320, "f16", None, seed=4)
    _gemv_check(lqm, handle, p0, lqm.FMT_2BIT, xb, "f16")
    p1 = O.quantize_2bit(W, np.arange(64, 96, dtype=np.int32))     # one whole group anchored
    _gemv_check(lqm, handle, p1, lqm.FMT_2BIT, xb, "f16")


def test_gemv_deterministic(lqm, handle):
    N, K = 700, 11008
    p, outl = quantized_2bit(N, K, seed=8)
    w = lqm.QuantWeights.from_host(p, lqm.FMT_2BIT)
    x = dev_x(x_for(1, K, "f16", outl, seed=8), "f16")
    ys = [handle.gemv(w, x).cpu() for _ in range(3)]
    assert all(torch.equal(ys[0], y) for y in ys[1:])


# ---------------------------------------------------------------- grouped and batched launches

def test_gemv_grouped_layer_small(lqm, handle):
    shapes = [(96, 512), (96, 512), (200, 512), (96, 1024)]
    probs, refs, ys = [], [], []
    for i, (N, K) in enumerate(shapes):
        p, outl = quantized_2bit(N, K, seed=40 + i)
        w = lqm.QuantWeights.from_host(p, lqm.FMT_2BIT)
        xb = x_for(4, K, "f16", outl, seed=40 + i)
        x = dev_x(xb, "f16")
        y = torch.empty((4, N), dtype=torch.float32, device="cuda")
        probs.append(handle.problem(w, x, y))
        refs.append((O.matmul_ref(O.dequant_2bit(p), xb, "f16"), w, x))
        ys.append(y)
    handle.gemv_grouped(probs)
    torch.cuda.synchronize()
    for (yref, E), y in zip([r[0] for r in refs], ys):
        assert_within(y.cpu().numpy(), yref, E, GEMV_TOL, "grouped")


def test_gemv_batched_distinct_weight_sets(lqm, handle):
    """512x256 single-linear problems, L distinct seeded weight sets in one launch."""
    L, N, K = 6, 512, 256
    packs = []
    for l in range(L):
        W = synth.weights(N, K, 0.02, seed=l, cfg=1)
        packs.append(O.quantize_2bit(W, O.select_anchors(W, O.activation_profile(np.ones(K)))))
    xs = [synth.activations(1, K, "f16", seed=l, cfg=1) for l in range(L)]
    stack = lambda key: np.stack([p[key] for p in packs])
    big = dict(codes=stack("codes"), scales=stack("scales"), offsets=stack("offsets"), anchor_idx=stack("anchor_idx"),
               anchor_w=stack("anchor_w"), A=packs[0]["A"], ld_anchor=packs[0]["ld_anchor"], N=N, K=K)
    w = lqm.QuantWeights.from_host(big, lqm.FMT_2BIT)
    x = dev_x(np.stack(xs), "f16")                                  # [L][1][K]
    y = torch.empty((L, 1, N), dtype=torch.float32, device="cuda")
    strides = dict(codes=N * K // 4, scales=N * K // 32 * 2, offsets=N * K // 32 * 2, anchor_idx=4 * big["A"],
                   anchor_w=N * big["ld_anchor"] * 2, x=K * 2, y=N * 4)
    if strides["anchor_idx"] % 16:
        pytest.skip("anchor_idx stride not 16-byte aligned for this A")
    handle.gemv_grouped([handle.problem(w, x[0], y[0], batch=L, strides=strides)])
    torch.cuda.synchronize()
    for l in range(L):
        yref, E = O.matmul_ref(O.dequant_2bit(packs[l]), xs[l], "f16")
        assert_within(y[l].cpu().numpy(), yref, E, GEMV_TOL, f"batch member {l}")


def test_gemv_512x256_batched_full_size_sampled(lqm, handle):
    """The 512x256 single linear as the bench runs it: 32768 distinct weight sets in one launch."""
    L, N, K, A = 32768, 512, 256, 8
    big = synth.random_packed_2bit_sets(L, N, K, A, seed=11, cfg=1)
    w = lqm.QuantWeights.from_host(big, lqm.FMT_2BIT)
    xb = synth.activations(L, K, "f16", seed=11, cfg=1)
    x = dev_x(xb.reshape(L, 1, K), "f16")
    y = torch.empty((L, 1, N), dtype=torch.float32, device="cuda")
    strides = dict(codes=N * K // 4, scales=N * K // 32 * 2, offsets=N * K // 32 * 2, anchor_idx=4 * A,
                   anchor_w=N * big["ld_anchor"] * 2, x=K * 2, y=N * 4)
    handle.gemv_grouped([handle.problem(w, x[0], y[0], batch=L, strides=strides)])
    yc = y.cpu().numpy()
    g = np.random.default_rng(3)
    for l in sorted(set(g.choice(L, 6, replace=False).tolist()) | {0, L - 1}):
        one = {k: (v[l] if isinstance(v, np.ndarray) else v) for k, v in big.items()}
        xl = xb[l:l + 1]
        yref = O.gemv_2bit_rows(one, xl, "f16", 0, N)
        E = O.row_error_scale(O.dequant_2bit(one), xl, "f16")
        assert_within(yc[l], yref, E, GEMV_TOL, f"set {l}")


# ---------------------------------------------------------------- full workload sizes, sampled rows

def _sampled_rows(N, k=24, seed=0):
    g = np.random.default_rng(seed)
    rows = set(g.choice(N, size=min(k, N), replace=False).tolist()) | {0, N - 1}
    return sorted(rows)


def _check_sampled_2bit(packed, xbits, xdt, y, rows, tol=GEMV_TOL, what=""):
    for n in rows:
        yr = O.gemv_2bit_rows(packed, xbits, xdt, n, n + 1)
        one = {k: (v[n:n + 1] if k in ("codes", "scales", "offsets", "anchor_w") else v) for k, v in packed.items()}
        one["N"] = 1
        E = O.row_error_scale(O.dequant_2bit(one), xbits, xdt)
        assert_within(y[:, n:n + 1], yr, E, tol, f"{what} row {n}")


@pytest.mark.parametrize("layer,M", [("7b", 1), ("70b", 1), ("70b", 8), ("70b", 32)])
def test_gemv_full_layer_sampled(lqm, handle, layer, M):
    """The bench's launch: one grouped call over a whole decoder layer at full size."""
    sigma = 0.02 if layer == "7b" else 0.015
    probs, keep = [], []
    for i, (name, N, K) in enumerate(synth.LAYER_SHAPES[layer]):
        A = O.anchor_count(K)
        pk = synth.random_packed_2bit(N, K, A, sigma=sigma, seed=1, cfg=2, matrix_id=i)
        w = lqm.QuantWeights.from_host(pk, lqm.FMT_2BIT)
        xb = synth.activations(M, K, "f16", synth.channel_sigma(K, synth.outlier_channels(K, 0.01, seed=1)), seed=1,
                               matrix_id=i)
        x = dev_x(xb, "f16")
        y = torch.empty((M, N), dtype=torch.float32, device="cuda")
        probs.append(handle.problem(w, x, y))
        keep.append((pk, xb, y, w, x))
    handle.gemv_grouped(probs)
    torch.cuda.synchronize()
    for i, (pk, xb, y, _, _) in enumerate(keep):
        _check_sampled_2bit(pk, xb, "f16", y.cpu().numpy(), _sampled_rows(pk["N"], 8, seed=i), what=f"{layer}[{i}]")


@pytest.mark.parametrize("M", [1, 4, 16])
def test_gemv_nf4_full_layer_sampled(lqm, handle, M):
    probs, keep = [], []
    for i, (name, N, K) in enumerate(synth.LAYER_SHAPES["7b"]):
        pk = synth.random_packed_nf4(N, K, seed=3, cfg=3, matrix_id=i)
        w = lqm.QuantWeights.from_host(pk, lqm.FMT_NF4)
        xb = synth.activations(M, K, "bf16", None, seed=3, matrix_id=i)
        x = dev_x(xb, "bf16")
        y = torch.empty((M, N), dtype=torch.float32, device="cuda")
        probs.append(handle.problem(w, x, y))
        keep.append((pk, xb, y, w, x))
    handle.gemv_grouped(probs)
    torch.cuda.synchronize()
    for i, (pk, xb, y, _, _) in enumerate(keep):
        yc = y.cpu().numpy()
        for n in _sampled_rows(pk["N"], 6, seed=i):
            yr = O.gemv_nf4_rows(pk, xb, "bf16", n, n + 1)
            one = dict(codes=pk["codes"][n:n + 1], absmax=pk["absmax"][n:n + 1], N=1, K=pk["K"])
            E = O.row_error_scale(O.dequant_nf4(one), xb, "bf16")
            assert_within(yc[:, n:n + 1], yr, E, GEMV_TOL, f"nf4[{i}] row {n}")


# ---------------------------------------------------------------- error paths on a live device

def test_errors_on_device_launch_nothing(lqm, handle):
    import ctypes
    p, _ = quantized_2bit(64, 256, seed=1)
    w = lqm.QuantWeights.from_host(p, lqm.FMT_2BIT)
    x = dev_x(x_for(1, 256, "f16"), "f16")
    with pytest.raises(lqm.LQError) as e:
        handle.gemv(w, torch.zeros((33, 256), dtype=torch.float16, device="cuda"))
    assert e.value.status == lqm.LQ_ERR_UNSUPPORTED
    y = torch.full((1, 64), 7.0, device="cuda")
    L = lqm.load_library()
    st = L.lq_gemv(handle.raw, 1, w.codes.data_ptr() + 1, w.scales.data_ptr(), w.offsets.data_ptr(),
                   w.anchor_idx.data_ptr(), w.anchor_w.data_ptr(), w.A, w.ld_anchor, x.data_ptr(), 1, y.data_ptr(), 0,
                   1, 64, 256, None)
    assert st == lqm.LQ_ERR_ALIGNMENT
    torch.cuda.synchronize()
    assert torch.all(y == 7.0)               # nothing ran
    handle.sync()


# ---------------------------------------------------------------- both decode kernels on the same shapes

@pytest.mark.parametrize("kernel", ["regs", "stream", "ring"])
@pytest.mark.parametrize("M", [1, 8, 9, 32])
def test_gemv_kernel_choice_same_results(lqm, handle, monkeypatch, kernel, M):
    """The split-K, the streaming and the ring kernels each meet the bound on a K % 256 == 0
    shape, for token counts on both sides of the default switch between the last two."""
    monkeypatch.setenv("LQ_GEMV_KERNEL", kernel)
    N, K = 300, 3072
    p, outl = quantized_2bit(N, K, seed=50 + M)
    xb = x_for(M, K, "f16", outl, seed=50 + M)
    _gemv_check(lqm, handle, p, lqm.FMT_2BIT, xb, "f16")
    pn = quantized_nf4(N, K, seed=60 + M)
    xn = x_for(M, K, "bf16", None, seed=60 + M)
    _gemv_check(lqm, handle, pn, lqm.FMT_NF4, xn, "bf16")


@pytest.mark.parametrize("M", [1, 4, 16])
def test_gemv_in_kernel_x_build(lqm, handle, monkeypatch, M):
    """LQ_GEMV_STAGE=1: the CTAs build the fragment-ordered x in shared memory (no pre-pass)."""
    monkeypatch.setenv("LQ_GEMV_STAGE", "1")
    for i, (N, K) in enumerate([(300, 3072), (80, 256)]):
        p, outl = quantized_2bit(N, K, seed=70 + M + i)
        xb = x_for(M, K, "f16", outl, seed=70 + M + i)
        _gemv_check(lqm, handle, p, lqm.FMT_2BIT, xb, "f16")
        pn = quantized_nf4(N, K, seed=80 + M + i)
        xn = x_for(M, K, "bf16", None, seed=80 + M + i)
        _gemv_check(lqm, handle, pn, lqm.FMT_NF4, xn, "bf16")


def test_gemv_full_projection_quantized_by_the_oracle(lqm, handle):
    """A full 4096 x 4096 projection quantized by the oracle from the listed distribution
    (profile-guided anchors on the x20 outlier channels), M = 1, every output checked."""
    N = K = 4096
    p, outl = quantized_2bit(N, K, seed=12, cfg=2)
    assert set(outl.tolist()) <= set(p["anchor_idx"].tolist())
    xb = x_for(1, K, "f16", outl, seed=12, cfg=2)
    _gemv_check(lqm, handle, p, lqm.FMT_2BIT, xb, "f16")


@pytest.mark.parametrize("A", [1, 7, 8, 15, 16, 17, 48, 49])
@pytest.mark.parametrize("M", [1, 5])
def test_gemv_anchor_counts_around_the_fused_limit(lqm, handle, A, M):
    """Up to 16 anchors ride in the last code unit of each row block (no anchor units); 17
    and more take anchor units of 48 columns.  Anchor counts on both sides of both limits,
    2-bit and INT4, on a shape with a ragged row block."""
    N, K = 150, 512
    W = synth.weights(N, K, 0.02, seed=A, big_frac=0.002, big_mult=10.0)
    prof = O.activation_profile(np.linspace(0.5, 3.0, K))
    ai = O.select_anchors(W, prof, frac=(A + 0.5) / K)
    assert len(ai) == A
    xb = x_for(M, K, "f16", seed=A + M)
    p2 = O.quantize_2bit(W, ai)
    _gemv_check(lqm, handle, p2, lqm.FMT_2BIT, xb, "f16")
    p4 = O.quantize_int4(W, O.int4_permutation(W, prof), ai)
    w4 = lqm.QuantWeights.from_host(p4, lqm.FMT_INT4)
    y = handle.gemv(w4, dev_x(xb, "f16"), y_dtype=torch.float32)
    torch.cuda.synchronize()
    yref, E = O.matmul_ref(O.dequant_int4(p4), xb, "f16")
    assert_within(y.cpu().numpy(), yref, E, GEMV_TOL, f"int4 A={A} M={M}")
    handle.sync()
