"""The timeout path of the kernels' bounded waits, run on the GPU without a fault:
a wait on a barrier that nothing completes gives up after its limit, raises the
handle's status word, and lq_sync reports LQ_ERR_TIMEOUT; the context stays usable
and the next calls compute correctly."""
import pytest

from oracle import oracle as O
from tests._util import assert_within, quantized_2bit, x_for

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lqm():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import bit_weight_quantized_dequant_gb300 as lq
    lq.build()
    return lq


def test_bounded_wait_reports_timeout_and_recovers(lqm):
    h = lqm.Handle(0)
    try:
        h.sync()                                  # clean to start with
        h.selftest_wait(20_000)                   # 20 ms
        with pytest.raises(lqm.LQError) as e:
            h.sync()
        assert e.value.status == lqm.LQ_ERR_TIMEOUT
        h.sync()                                  # the flag was cleared
        # the handle still computes correctly after the timeout
        p, outl = quantized_2bit(200, 1024, seed=3)
        w = lqm.QuantWeights.from_host(p, lqm.FMT_2BIT)
        xb = x_for(4, 1024, "f16", outl, seed=3)
        y = h.gemv(w, torch.from_numpy(xb).view(torch.float16).cuda())
        h.sync()
        yref, E = O.matmul_ref(O.dequant_2bit(p), xb, "f16")
        assert_within(y.cpu().numpy(), yref, E, 1e-3, "gemv after a timeout")
    finally:
        h.close()
