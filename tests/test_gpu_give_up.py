"""The bounded-wait give-up path of the skinny kernels, on the GPU, without
faulting or hanging it.

A test shortens the wait limit (wq_debug_set_wait_limit) to 1 ns, so that the
first wait whose data has not landed yet gives up (L2 is flushed first, so
the weights come from HBM): the kernel records its site
in the device error word, every warp leaves its loop, the copies in flight are
drained, and the call returns.  wq_get_device_error then reports WQ_ERR_DEVICE
with the consumer-wait site, and with the default limit restored the next call
on the same stream computes the right result (the context is still usable)."""
import pytest

import workloads
from oracle import wq_oracle as O
from tests.gpu_util import assert_gemm_close

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

SITE_CONSUMER_WAIT = 2  # kSiteGemmMma: a consumer waited too long for its data


@pytest.fixture(scope="module")
def wq():
    import bit_quantized_gemm_dequant_gb300 as mod

    return mod


def _flush_l2():
    """Overwrite more than the 129 MB L2, so that the weights come from HBM and
    the waits find their data still in flight."""
    torch.empty(64 << 20, dtype=torch.float32, device="cuda").fill_(1.0)


def _give_up_then_recover(wq, call, check):
    assert wq.wq_get_device_error() == (wq.WQ_OK, 0)
    try:
        wq.wq_debug_set_wait_limit(1)
        _flush_l2()
        call()
        torch.cuda.synchronize()
    finally:
        wq.wq_debug_set_wait_limit(0)
    st, site = wq.wq_get_device_error()
    assert st == wq.WQ_ERR_DEVICE and site == SITE_CONSUMER_WAIT
    assert wq.wq_get_device_error() == (wq.WQ_OK, 0)  # read and cleared
    check(call())
    torch.cuda.synchronize()
    assert wq.wq_get_device_error() == (wq.WQ_OK, 0)


def test_per_call_kernel_gives_up_and_recovers(wq):
    # 1 x 4096 x 14336: one CTA per 128-column tile, no workspace hand-shake.
    c = workloads.w8a16_case(1, 4096, 14336, seed=3)
    x, w, s = (torch.from_numpy(a).cuda() for a in (c.x, c.w, c.scales))
    _give_up_then_recover(wq, lambda: wq.wq_gemm_w8a16(x, w, s),
                          lambda y: assert_gemm_close(y, O.gemm_w8a16(c.x, c.w, c.scales), "fp16"))


def test_batched_kernel_gives_up_and_recovers(wq):
    cases = [workloads.w4a16_case(1, 4096, 4096, seed=4), workloads.w4a16_case(8, 4096, 11008, seed=5)]
    xs = [torch.from_numpy(c.x).cuda() for c in cases]
    ws = [torch.from_numpy(c.w).cuda() for c in cases]
    ss = [torch.from_numpy(c.scales).cuda() for c in cases]
    ws_buf = torch.zeros(8 << 20, dtype=torch.uint8, device="cuda")

    def check(ys):
        for c, y in zip(cases, ys):
            assert_gemm_close(y, O.gemm_w4a16(c.x, c.w, c.scales), "fp16")

    def call():
        return wq.wq_gemm_w4a16_batched(xs, ws, ss, workspace=ws_buf)

    assert wq.wq_get_device_error() == (wq.WQ_OK, 0)
    try:
        wq.wq_debug_set_wait_limit(1)
        _flush_l2()
        call()
        torch.cuda.synchronize()
    finally:
        wq.wq_debug_set_wait_limit(0)
    st, site = wq.wq_get_device_error()
    assert st == wq.WQ_ERR_DEVICE and site in (SITE_CONSUMER_WAIT, 6)  # 6: a finalizer gave up on a neighbour
    ws_buf.zero_()  # after WQ_ERR_DEVICE the workspace is zeroed again before reuse
    check(call())
    torch.cuda.synchronize()
    assert wq.wq_get_device_error() == (wq.WQ_OK, 0)
