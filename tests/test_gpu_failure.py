"""Failure detection on the GPU without a fault: a kernel's bounded wait on a
barrier that nothing arrives on gives up, the host reads WL_ERR_TIMEOUT from
the device status word (then the word is clear), and the context still
computes correctly."""
import pytest
import torch

import wl_synth
from tests.parity import assert_parity

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout(wl, orc, gpu):
    assert wl.wl_device_status() == wl.WL_OK  # nothing pending from earlier tests
    wl.wl_selftest_wait()
    assert wl.wl_device_status() == wl.WL_ERR_TIMEOUT
    assert "ring-full" in wl.wl_last_error()
    assert wl.wl_device_status() == wl.WL_OK  # read and cleared
    x, th = wl_synth.linear_case(12, 4, 1152, 1024, 4)
    tg = th.to(gpu)
    y = wl.wl_linear(x.to(gpu), tg.W0, tg.s, tg.U, tg.V)
    torch.cuda.synchronize()
    assert wl.wl_device_status() == wl.WL_OK
    assert_parity(y, orc.linear(x, th), torch.bfloat16, "after the timeout")
