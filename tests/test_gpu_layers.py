"""GPU parity of lq_gemv_layers: consecutive decode layers in one call, where a layer reads, as x,
what the layer before it wrote.

* The call's outputs equal, bit for bit, one lq_gemv_grouped call per layer in order, so a
  layer that ran before its input was complete would show up as a mismatch.
* Every layer's outputs are within the GEMV bound of the oracle applied to that layer's actual
  input (read back from the GPU): |y - y_ref| <= 1e-3 * sum_k |W_eff||x|, plus one binary16
  rounding (2^-11 |y_ref|) where the layer writes binary16 for the next layer to read.
* 2-bit, INT4 and NF4 layers, a layer on the split-K kernel, and 7B-shaped layers.
"""
import numpy as np
import pytest

import synth
from oracle import oracle as O
from tests._util import quantized_2bit, quantized_int4, quantized_nf4, x_for

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

GEMV_TOL = 1e-3
HALF_ROUND = 2.0 ** -11


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


def bits(t):
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


def check_layer(y, yref, E, half_out, what):
    y = np.asarray(y, dtype=np.float64)
    bound = GEMV_TOL * E + (HALF_ROUND * np.abs(yref) if half_out else 0.0) + 1e-30
    err = np.abs(y - yref)
    assert np.all(err <= bound), f"{what}: max err/bound {np.max(err / bound):.3f}"


class Chain:
    """Layers of (weights, dequantized oracle weights, N, K, source) where source is ("in", bits)
    for a given input or ("y", layer, index) for an earlier layer's output."""

    def __init__(self, lqm, handle, fmt):
        self.lqm, self.h, self.fmt, self.layers = lqm, handle, fmt, []

    def add_layer(self, items):
        self.layers.append(items)

    def build(self, last_f32=True):
        """Problems over fresh output buffers: binary16 outputs, except the last layer's."""
        ys, probs = [], []
        for li, items in enumerate(self.layers):
            last = li == len(self.layers) - 1
            ly, lp = [], []
            for (w, Wd, N, K, src) in items:
                x = src[1] if src[0] == "in" else ys[src[1]][src[2]]
                y = torch.empty((1, N), dtype=torch.float32 if (last and last_f32) else torch.float16, device="cuda")
                ly.append(y)
                lp.append(self.h.problem(w, x, y))
            ys.append(ly)
            probs.append(lp)
        return probs, ys

    def check_oracle(self, ys, what):
        for li, items in enumerate(self.layers):
            for i, (w, Wd, N, K, src) in enumerate(items):
                xb = bits(src[1]) if src[0] == "in" else bits(ys[src[1]][src[2]])
                yref, E = O.matmul_ref(Wd, xb.reshape(1, K), "f16")
                y = ys[li][i]
                check_layer(y.float().cpu().numpy(), yref, E, y.dtype == torch.float16, f"{what} layer {li}[{i}]")


def _input(K, seed):
    xb = x_for(1, K, "f16", None, seed=seed)
    return torch.from_numpy(np.ascontiguousarray(xb)).view(torch.float16).cuda()


def _run_both(chain):
    p1, y1 = chain.build()
    chain.h.gemv_layers(p1)
    torch.cuda.synchronize()
    p2, y2 = chain.build()
    for layer in p2:
        chain.h.gemv_grouped(layer)
    torch.cuda.synchronize()
    for a, b in zip(y1, y2):
        for ya, yb in zip(a, b):
            assert torch.equal(ya, yb), "lq_gemv_layers and one grouped call per layer differ"
    return p1, y1


def _small_2bit(lqm, handle):
    c = Chain(lqm, handle, lqm.FMT_2BIT)

    def mk(N, K, seed, src):
        p, _ = quantized_2bit(N, K, seed=seed)
        return (lqm.QuantWeights.from_host(p, lqm.FMT_2BIT), O.dequant_2bit(p), N, K, src)

    c.add_layer([mk(512, 512, 60, ("in", _input(512, 1))), mk(256, 256, 61, ("in", _input(256, 2)))])
    c.add_layer([mk(256, 512, 62, ("y", 0, 0)), mk(512, 256, 63, ("y", 0, 1))])
    c.add_layer([mk(512, 256, 64, ("y", 1, 0)), mk(256, 512, 65, ("y", 1, 1))])
    c.add_layer([mk(768, 512, 66, ("y", 2, 0))])
    c.add_layer([mk(256, 768, 67, ("y", 3, 0)), mk(512, 256, 68, ("y", 2, 1))])
    return c


def test_layers_2bit_small_chain(lqm, handle):
    """Five 2-bit layers with cross-layer inputs."""
    c = _small_2bit(lqm, handle)
    _, ys = _run_both(c)
    c.check_oracle(ys, "2-bit")


def test_layers_repeated_calls_stay_in_step(lqm, handle):
    """Many calls back to back (launches overlapping at their edges): the same results."""
    c = _small_2bit(lqm, handle)
    probs, ys = c.build()
    handle.gemv_layers(probs)
    torch.cuda.synchronize()
    first = [[y.clone() for y in layer] for layer in ys]
    for _ in range(25):
        handle.gemv_layers(probs)
    torch.cuda.synchronize()
    handle.sync()
    for a, b in zip(first, ys):
        for ya, yb in zip(a, b):
            assert torch.equal(ya, yb)


def test_layers_int4_chain(lqm, handle):
    c = Chain(lqm, handle, lqm.FMT_INT4)

    def mk(N, K, seed, src):
        p, _ = quantized_int4(N, K, seed=seed)
        return (lqm.QuantWeights.from_host(p, lqm.FMT_INT4), O.dequant_int4(p), N, K, src)

    c.add_layer([mk(512, 512, 70, ("in", _input(512, 3)))])
    c.add_layer([mk(256, 512, 71, ("y", 0, 0)), mk(512, 512, 72, ("y", 0, 0))])
    c.add_layer([mk(512, 256, 73, ("y", 1, 0))])
    _, ys = _run_both(c)
    c.check_oracle(ys, "INT4")


def test_layers_nf4(lqm, handle):
    c = Chain(lqm, handle, lqm.FMT_NF4)

    def mk(N, K, seed, src):
        p = quantized_nf4(N, K, seed=seed)
        return (lqm.QuantWeights.from_host(p, lqm.FMT_NF4), O.dequant_nf4(p), N, K, src)

    c.add_layer([mk(256, 512, 80, ("in", _input(512, 4)))])
    c.add_layer([mk(512, 256, 81, ("y", 0, 0))])
    _, ys = _run_both(c)
    c.check_oracle(ys, "NF4")


def test_layers_with_a_split_k_layer(lqm, handle):
    """A layer whose K is not a multiple of 256 (split-K kernel) between ring-kernel layers."""
    c = Chain(lqm, handle, lqm.FMT_2BIT)

    def mk(N, K, seed, src):
        p, _ = quantized_2bit(N, K, seed=seed)
        return (lqm.QuantWeights.from_host(p, lqm.FMT_2BIT), O.dequant_2bit(p), N, K, src)

    c.add_layer([mk(384, 512, 90, ("in", _input(512, 7)))])
    c.add_layer([mk(512, 384, 91, ("y", 0, 0))])
    c.add_layer([mk(256, 512, 92, ("y", 1, 0))])
    _, ys = _run_both(c)
    c.check_oracle(ys, "split-K")


def _layer_7b(lqm, seed):
    ws = []
    for i, (name, N, K) in enumerate(synth.LAYER_SHAPES["7b"]):
        pk = synth.random_packed_2bit(N, K, O.anchor_count(K), sigma=0.02, seed=seed, cfg=2, matrix_id=i)
        ws.append((name, N, K, pk, lqm.QuantWeights.from_host(pk, lqm.FMT_2BIT)))
    return ws


def test_layers_7b_stack(lqm, handle):
    """Six 7B-shaped layers (the bench's decode step): the six K = 4096 projections of layer l + 1
    read layer l's down-projection output, and its down projection reads layer l's gate output.
    The call equals one grouped call per layer bit for bit; sampled rows of the last layer
    against the oracle on its actual inputs."""
    sets = [_layer_7b(lqm, s) for s in (11, 12)]
    names = [s[0] for s in sets[0]]
    i_down, i_gate = names.index("down"), names.index("gate")
    x0 = _input(4096, 5)
    xd0 = _input(11008, 6)

    def build():
        ys, probs = [], []
        for l in range(6):
            layer, ly = [], []
            for j, (name, N, K, pk, w) in enumerate(sets[l % 2]):
                if l == 0:
                    x = xd0 if name == "down" else x0
                else:
                    x = ys[l - 1][i_gate] if name == "down" else ys[l - 1][i_down]
                y = torch.empty((1, N), dtype=torch.float16, device="cuda")
                ly.append(y)
                layer.append(handle.problem(w, x, y))
            ys.append(ly)
            probs.append(layer)
        return probs, ys

    p1, y1 = build()
    handle.gemv_layers(p1)
    torch.cuda.synchronize()
    p2, y2 = build()
    for layer in p2:
        handle.gemv_grouped(layer)
    torch.cuda.synchronize()
    for a, b in zip(y1, y2):
        for ya, yb in zip(a, b):
            assert torch.equal(ya, yb)
    last = 5
    for j, (name, N, K, pk, w) in enumerate(sets[last % 2]):
        src = y1[last - 1][i_gate] if name == "down" else y1[last - 1][i_down]
        xb = bits(src).reshape(1, K)
        yc = y1[last][j].float().cpu().numpy()
        g = np.random.default_rng(j)
        for n in sorted(set(g.choice(N, size=6, replace=False).tolist()) | {0, N - 1}):
            yr = O.gemv_2bit_rows(pk, xb, "f16", n, n + 1)
            one = {k: (v[n:n + 1] if k in ("codes", "scales", "offsets", "anchor_w") else v) for k, v in pk.items()}
            one["N"] = 1
            E = O.row_error_scale(O.dequant_2bit(one), xb, "f16")
            check_layer(yc[:, n:n + 1], yr, E, True, f"7B layer {last} {name} row {n}")
