"""The decode launch's plan cache (a call with the same problems, workspace and kernel choice
reuses its launch description): results are those of a fresh plan, across evictions, across
calls of one kernel with different shared-memory sizes, and across a change of kernel choice."""
import numpy as np
import pytest

from oracle import oracle as O
from tests._util import assert_within, quantized_2bit, x_for

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


def _case(lqm, handle, N, K, M, seed):
    p, outl = quantized_2bit(N, K, seed=seed)
    w = lqm.QuantWeights.from_host(p, lqm.FMT_2BIT)
    xb = x_for(M, K, "f16", outl, seed=seed)
    x = torch.from_numpy(np.ascontiguousarray(xb)).view(torch.float16).cuda()
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    yref, E = O.matmul_ref(O.dequant_2bit(p), xb, "f16")
    return dict(w=w, x=x, y=y, yref=yref, E=E, prob=handle.problem(w, x, y))


def test_repeated_and_evicted_calls(lqm, handle):
    """20 distinct calls (more than the cache holds), then every one again: the same outputs."""
    cases = [_case(lqm, handle, 64 * (1 + i % 5), 256 * (1 + i % 3), 1 + i % 4, 200 + i) for i in range(20)]
    first = []
    for c in cases:
        handle.gemv_grouped([c["prob"]])
        torch.cuda.synchronize()
        assert_within(c["y"].cpu().numpy(), c["yref"], c["E"], GEMV_TOL, "fresh plan")
        first.append(c["y"].clone())
    for rep in range(2):
        for c, y0 in zip(cases, first):
            c["y"].zero_()
            handle.gemv_grouped(handle.prepare([c["prob"]]))
            torch.cuda.synchronize()
            assert torch.equal(c["y"], y0)


def test_one_kernel_two_shared_memory_sizes(lqm, handle):
    """Calls of the same kernel instantiation whose x spans (shared memory) differ, alternating:
    each launch keeps a valid shared-memory attribute."""
    small = _case(lqm, handle, 256, 256, 1, 301)
    big = [_case(lqm, handle, 64, 4096, 1, 302 + i) for i in range(3)]
    p_small, p_big = handle.prepare([small["prob"]]), handle.prepare([c["prob"] for c in big])
    for _ in range(4):
        handle.gemv_grouped(p_big)
        handle.gemv_grouped(p_small)
    torch.cuda.synchronize()
    handle.sync()
    for c in [small] + big:
        assert_within(c["y"].cpu().numpy(), c["yref"], c["E"], GEMV_TOL, "alternating sizes")


def test_kernel_choice_is_part_of_the_key(lqm, handle, monkeypatch):
    c = _case(lqm, handle, 320, 1024, 4, 310)
    outs = []
    for kern in ("ring", "stream", "ring"):
        monkeypatch.setenv("LQ_GEMV_KERNEL", kern)
        c["y"].zero_()
        handle.gemv_grouped([c["prob"]])
        torch.cuda.synchronize()
        assert_within(c["y"].cpu().numpy(), c["yref"], c["E"], GEMV_TOL, kern)
        outs.append(c["y"].clone())
    assert torch.equal(outs[0], outs[2])
