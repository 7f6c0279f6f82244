"""GPU tests of layer streaming (lq_stream_run): a stack whose packed weights live in
pinned host memory, copied layer by layer into two device slots while the previous
layer computes.  Each layer's output equals, bit for bit, the same grouped GEMV run
on device-resident copies of that layer (same kernels, same launch shape), and meets
the oracle's bound."""
import numpy as np
import pytest

import synth
from oracle import oracle as O
from tests._util import assert_within

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

SHAPES = [(300, 1024), (128, 512), (64, 2048)]


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


def make_stack(lqm, fmt, L, seed=0):
    layers = []
    for l in range(L):
        packs = []
        for i, (N, K) in enumerate(SHAPES):
            if fmt == lqm.FMT_2BIT:
                packs.append(synth.random_packed_2bit(N, K, O.anchor_count(K), seed=seed + l, cfg=2, matrix_id=i))
            else:
                packs.append(synth.random_packed_nf4(N, K, seed=seed + l, cfg=3, matrix_id=i))
        layers.append(packs)
    blobs = [lqm.pack_layer(p, fmt) for p in layers]
    layer_bytes = max(b.nbytes for b, _ in blobs)
    stride = (layer_bytes + 4095) // 4096 * 4096
    host = torch.empty(L * stride, dtype=torch.uint8).pin_memory()
    hv = host.numpy()
    for l, (b, _) in enumerate(blobs):
        hv[l * stride:l * stride + b.nbytes] = b
    return layers, blobs[0][1], host, stride, layer_bytes


@pytest.mark.parametrize("fmt_name", ["2bit", "nf4"])
@pytest.mark.parametrize("M", [1, 4])
def test_stream_equals_resident_layers(lqm, handle, fmt_name, M):
    fmt = lqm.FMT_2BIT if fmt_name == "2bit" else lqm.FMT_NF4
    L = 5
    layers, meta, host, stride, layer_bytes = make_stack(lqm, fmt, L, seed=10 * M)
    xdt = torch.float16 if fmt == lqm.FMT_2BIT else torch.bfloat16
    g = torch.Generator(device="cuda")
    g.manual_seed(M)
    xs = [torch.randn((M, K), generator=g, device="cuda").to(xdt) for (_, K) in SHAPES]
    ystride = max(M * N * 4 for (N, _) in SHAPES)
    ystride = (ystride + 255) // 256 * 256
    ys = [torch.zeros((L, ystride // 4), dtype=torch.float32, device="cuda") for _ in SHAPES]
    ls = lqm.LayerStream(handle, stride)
    probs = [ls.problem(meta[i], fmt, xs[i], ys[i]) for i in range(len(SHAPES))]
    for _ in range(2):   # a second pass reuses the slots
        ls.run(host, stride, layer_bytes, L, probs, y_layer_stride=ystride)
        torch.cuda.synchronize()
        for l in range(L):
            ws = [lqm.QuantWeights.from_host(p, fmt) for p in layers[l]]
            yr = [torch.empty((M, N), dtype=torch.float32, device="cuda") for (N, _) in SHAPES]
            handle.gemv_grouped([handle.problem(w, x, y) for w, x, y in zip(ws, xs, yr)])
            torch.cuda.synchronize()
            for i, (N, _) in enumerate(SHAPES):
                assert torch.equal(ys[i][l, :M * N].view(M, N), yr[i]), (l, i)
    ls.close()
    # and against the oracle (last layer, first matrix)
    p = layers[L - 1][0]
    Weff = O.dequant_2bit(p) if fmt == lqm.FMT_2BIT else O.dequant_nf4(p)
    xb = xs[0].cpu().view(torch.int16).numpy().view(np.uint16)
    yref, E = O.matmul_ref(Weff, xb, "f16" if fmt == lqm.FMT_2BIT else "bf16")
    assert_within(ys[0][L - 1, :M * SHAPES[0][0]].view(M, -1).cpu().numpy(), yref, E, 1e-3, "streamed layer")


@pytest.mark.parametrize("fmt_name,M", [("2bit", 1), ("nf4", 4)])
def test_stream_direct_equals_resident_layers(lqm, handle, fmt_name, M):
    """Kernels reading the pinned host bytes directly give the resident results bit for bit."""
    fmt = lqm.FMT_2BIT if fmt_name == "2bit" else lqm.FMT_NF4
    L = 4
    layers, meta, host, stride, layer_bytes = make_stack(lqm, fmt, L, seed=7 + M)
    xdt = torch.float16 if fmt == lqm.FMT_2BIT else torch.bfloat16
    xs = [torch.randn((M, K), device="cuda").to(xdt) for (_, K) in SHAPES]
    ystride = (max(M * N * 4 for (N, _) in SHAPES) + 255) // 256 * 256
    ys = [torch.zeros((L, ystride // 4), dtype=torch.float32, device="cuda") for _ in SHAPES]
    ls = lqm.LayerStream(handle, 256)
    probs = [ls.problem(meta[i], fmt, xs[i], ys[i]) for i in range(len(SHAPES))]
    try:
        ls.run_direct(host, stride, layer_bytes, L, probs, y_layer_stride=ystride)
    except lqm.LQError as e:
        if e.status == lqm.LQ_ERR_UNSUPPORTED:
            pytest.skip("pinned memory without a device mapping on this system")
        raise
    torch.cuda.synchronize()
    for l in range(L):
        ws = [lqm.QuantWeights.from_host(p, fmt) for p in layers[l]]
        yr = [torch.empty((M, N), dtype=torch.float32, device="cuda") for (N, _) in SHAPES]
        handle.gemv_grouped([handle.problem(w, x, y) for w, x, y in zip(ws, xs, yr)])
        torch.cuda.synchronize()
        for i, (N, _) in enumerate(SHAPES):
            assert torch.equal(ys[i][l, :M * N].view(M, N), yr[i]), (l, i)
    # memory the device has no mapping for (plain pageable host memory) is refused before any launch
    pageable = torch.empty(host.numel(), dtype=torch.uint8)
    assert not pageable.is_pinned()
    with pytest.raises(lqm.LQError) as e:
        ls.run_direct(pageable, stride, layer_bytes, L, probs, y_layer_stride=ystride)
    assert e.value.status == lqm.LQ_ERR_UNSUPPORTED
    ls.close()


def test_stream_rejects_before_copying(lqm, handle):
    layers, meta, host, stride, layer_bytes = make_stack(lqm, lqm.FMT_2BIT, 2)
    x = torch.zeros((1, SHAPES[0][1]), dtype=torch.float16, device="cuda")
    y = torch.zeros((1, SHAPES[0][0]), dtype=torch.float32, device="cuda")
    ls = lqm.LayerStream(handle, layer_bytes - 256)
    prob = ls.problem(meta[0], lqm.FMT_2BIT, x, y)
    with pytest.raises(lqm.LQError) as e:
        ls.run(host, stride, layer_bytes, 2, [prob])            # the layer does not fit a slot
    assert e.value.status == lqm.LQ_ERR_WORKSPACE
    bad = ls.problem(dict(meta[0], codes=layer_bytes), lqm.FMT_2BIT, x, y)   # codes past the layer
    with pytest.raises(lqm.LQError) as e:
        ls.run(host, stride, layer_bytes - 256, 1, [bad])
    assert e.value.status == lqm.LQ_ERR_INVALID_ARG
    ls.close()
