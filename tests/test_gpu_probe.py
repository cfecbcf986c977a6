"""The diagnostic FP32-pipe probe runs one CTA per SM and writes its sink."""
import pytest
import torch

import gated_deltanet_linear_gdr_gb300 as gdr

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("pattern", [0, 1, 2])
def test_probe_fma_runs_one_cta_per_sm(pattern):
    dev = torch.device("cuda:0")
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    sink = torch.full((sms * 128 * 2,), float("nan"), device=dev)
    ctas = gdr.gdr_probe_fma(pattern, 1, 4, sink)
    torch.cuda.synchronize()
    assert ctas == sms
    assert torch.isfinite(sink[: sms * 128]).all()
    assert gdr.gdr_get_status(clear=True) == 0


def test_probe_fma_rejects_a_short_sink():
    dev = torch.device("cuda:0")
    sink = torch.empty(16, device=dev)
    with pytest.raises(gdr.GdrError):
        gdr.gdr_probe_fma(1, 1, 4, sink)
