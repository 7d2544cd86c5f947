"""Failure detection on the GPU without a fault: a bounded wait that nothing
completes gives up, the sticky device error word reports BI_ERR_TIMEOUT to
the host, reading it clears it, and the context keeps working."""
import time

import numpy as np
import pytest

from serving_numerics_gb300 import synth
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives(bi, orc):
    import torch
    assert bi.bi_get_last_device_error() == bi.BI_OK            # start clean
    t = time.perf_counter()
    assert bi.bi_selftest_wait_timeout(20000) == bi.BI_OK       # 20 ms bound
    assert bi.bi_get_last_device_error() == bi.BI_ERR_TIMEOUT
    elapsed = time.perf_counter() - t
    assert 0.015 < elapsed < 5.0
    assert bi.bi_get_last_device_error() == bi.BI_OK            # read clears it
    # the context is usable: a normal router call still matches the oracle
    X = synth.tokens(50, 0, 0, 8, 256)
    W = synth.router_weights(50, 0, 64, 256)
    out = bi.router_topk(gu.dev_f32(X), gu.dev_f32(W), 4, "f32")
    torch.cuda.synchronize()
    sel = orc.selection_from_logits(out["logits"].cpu().numpy(), 4)
    assert np.array_equal(out["ids"].cpu().numpy(), sel["ids"])
    assert bi.bi_get_last_device_error() == bi.BI_OK


def test_selftest_rejects_bad_limits(bi):
    assert bi.bi_selftest_wait_timeout(0) == bi.BI_ERR_INVALID_ARG
    assert bi.bi_selftest_wait_timeout(2000001) == bi.BI_ERR_INVALID_ARG
