"""The bounded copy wait of the staged kernels, made to run out.

Every staged kernel waits for its shared-memory copies with a wall-clock
limit and, when the limit passes, raises FP8Q_DEVICE_ERR_COPY_TIMEOUT and
returns rather than hanging or handing back silent garbage ("perf: Reduce
MXFP8 refit weight-transfer overheads", Safety: fail loudly).  A copy that
never lands cannot be caused on purpose without faulting the GPU, so the
library's self-test kernel arms a barrier for 16 bytes and issues no copy:
the same wait and the same give-up path then run out after a short limit,
with nothing in flight.  The tests check that the wait ran its limit, that
the error bit reaches the host, that it clears, and that the next ordinary
call still matches the oracle bit for bit."""
import numpy as np
import pytest
import torch

import gen
from gpu_util import bits16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def w():
    import weight_transfer_gb300 as w
    return w


def timed_ms(fn):
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    fn()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b)


@pytest.mark.parametrize("limit_ms", [10, 50])
def test_a_wait_that_never_completes_runs_out_reports_and_leaves_the_context_usable(w, orc, limit_ms):
    assert w.fp8q_device_errors(clear=True) == 0
    ms = timed_ms(lambda: w.fp8q_selftest_copy_wait(limit_ms * 1_000_000))
    assert ms >= 0.99 * limit_ms, f"gave up after {ms:.3f} ms, before its {limit_ms} ms limit"
    assert ms < 1000.0, f"took {ms:.1f} ms: the limit passed to the wait was not the one used"
    assert w.fp8q_device_errors(clear=True) == w.FP8Q_DEVICE_ERR_COPY_TIMEOUT
    assert w.fp8q_device_errors(clear=True) == 0                    # cleared
    # the next ordinary call runs normally and matches the oracle
    x = gen.normal_bf16(4096 * 8 + 77, 1e-3, seed=limit_ms, outlier_p=1e-3, outlier_mult=100.0)
    c, s = w.fp8q_quantize_blockwise(x.cuda(), "e4m3")
    ec, es = orc.quantize_blockwise(bits16(x), 0)
    assert np.array_equal(c.cpu().numpy(), ec)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), es.view(np.uint32))
    assert w.fp8q_device_errors(clear=False) == 0


def test_a_wait_whose_copy_lands_completes_without_an_error(w):
    src = torch.arange(16, dtype=torch.uint8, device="cuda").add_(100)
    dst = torch.zeros(16, dtype=torch.uint8, device="cuda")
    ms = timed_ms(lambda: w.fp8q_selftest_copy_wait(1_000_000_000, src, dst))
    assert torch.equal(dst, src)
    assert ms < 500.0                                                # did not wait out the 1 s limit
    assert w.fp8q_device_errors(clear=False) == 0
