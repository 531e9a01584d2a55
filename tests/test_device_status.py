"""The bounded-wait failure path on the GPU: a kernel whose barrier nothing completes gives up
after the wait limit, the host reads GCS_ERR_DEVICE_TIMEOUT from the device status word, and
the context stays usable for the next call (no fault, no hang)."""
import pytest
import torch

from synth import make_decode
from helpers import DECODE_RTOL, assert_close, oracle_decode, run_decode

pytestmark = pytest.mark.gpu

GCS_ERR_DEVICE_TIMEOUT = 5


def test_bounded_wait_times_out_and_context_stays_usable(gcs_lib):
    assert gcs_lib.get_device_status(clear=True) == 0
    assert gcs_lib.selftest_bounded_wait() == GCS_ERR_DEVICE_TIMEOUT
    # the word was cleared by the read; a normal call runs and reports no timeout
    assert gcs_lib.get_device_status(clear=False) == 0
    dc = make_decode([300, 2100], [1, 3], 16, 1, 128, seed=77)
    out = run_decode(gcs_lib, dc)
    assert_close("out", out, oracle_decode(dc), DECODE_RTOL)
    torch.cuda.synchronize()
