"""The device generator writes the same bits as the host generator."""
import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("spec", [
    synth.normal(1e-3, synth.BF16, synth.GRAD, 3, 7),
    synth.normal(1e-4, synth.BF16, synth.GRAD, 1, 1, outlier_every=100, outlier_mult=100.0),
    synth.uniform(6e-5, synth.FP16, synth.GRAD, 63, 1),
    synth.normal(0.02, synth.FP32, synth.MASTER),
    synth.normal(1e-8, synth.FP32, synth.MOM2, absolute=True),
])
def test_device_matches_host(spec):
    import torch

    for start, count in [(0, 1 << 20), ((1 << 33) + 12345, 100_003)]:
        t = torch.empty(count, dtype=torch.int32 if spec.fmt == synth.FP32 else torch.int16, device="cuda")
        synth.device_fill(spec, t, start=start)
        dev = t.cpu().numpy().view(np.uint32 if spec.fmt == synth.FP32 else np.uint16)
        assert np.array_equal(dev, synth.host_range(spec, start, count))
