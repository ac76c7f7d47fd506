"""Failure detection without a GPU fault: a kernel whose bounded wait can
never be satisfied must give up after its limit, report the timeout through
fa4fp4_sync_status, and leave the context usable."""
import time

import numpy as np
import pytest
import torch

from gpu_util import require_gpu

pytestmark = pytest.mark.gpu


def test_wait_that_never_completes_is_reported():
    fa = require_gpu()
    fa.sync_status()                       # clean start
    t0 = time.time()
    fa.watchdog_selftest(50_000_000)       # 50 ms
    with pytest.raises(fa.Fa4Fp4Error) as e:
        fa.sync_status()
    assert e.value.status == 5             # FA4FP4_ERR_DEVICE_TIMEOUT
    assert time.time() - t0 < 5.0
    fa.sync_status()                       # the flag was cleared
    # the context still runs work
    x = torch.randn(1, 1, 64, 64).to(torch.bfloat16).cuda()
    q = fa.quantize(x)
    fa.sync_status()
    assert q.scales.cpu().numpy().max() > 0


def test_selftest_argument_checks():
    fa = require_gpu()
    for bad in (0, -5, 3_000_000_000):
        with pytest.raises(fa.Fa4Fp4Error):
            fa.watchdog_selftest(bad)
