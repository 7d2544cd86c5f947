"""The FP32 FMA rate probe behind the router's ALU roofline: it runs, counts
the work it launches, and reports a rate in the range the GPU's FP32 lanes
allow (152 SMs x 128 lanes x 2 flop at 1-2.1 GHz is 39-81 TFLOP/s for
scalar FMAs; the two-wide instruction is allowed up to twice that).  A rate
far outside means the probe is not doing its work."""
import pytest

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("packed", [False, True])
def test_fma_probe_rate_is_plausible(bi, packed):
    import torch
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    sink = torch.empty((8 * sms,), dtype=torch.float32, device="cuda")
    flop = bi.selftest_fma_rate(2000, sink, packed=packed)
    assert flop == 2.0 * 8 * sms * 256 * 2000 * 16 * 8 * (2 if packed else 1)
    best = 0.0
    for _ in range(3):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        bi.selftest_fma_rate(2000, sink, packed=packed)
        b.record()
        torch.cuda.synchronize()
        best = max(best, flop / (a.elapsed_time(b) / 1e3) / 1e12)
    peak = sms * 128 * 2 * 2.2e9 / 1e12
    assert 0.3 * peak < best < (2.1 if packed else 1.05) * peak
    assert bi.bi_get_last_device_error() == bi.BI_OK
