"""mx_calibrate_mma: one wave of back-to-back block-scaled FP4 MMAs per SM (or
CTA pair), the tensor-pipe rate the benchmark reports as its per-clock ceiling.

Checked on the GPU: every form and shape completes with a clean status word,
every SM or pair reports its cycles, those cycles grow in proportion to the
number of MMAs (the per-MMA cost is a rate, not a start-up constant), and the
FLOP count the call reports is 2 M N K per MMA over the units it ran."""
import pytest
import torch

import block_scaled_fp4_bf16_gb300 as mx

pytestmark = pytest.mark.gpu

FORMS = [mx.MX_MMA_MXF4, mx.MX_MMA_MXF4NVF4_2X, mx.MX_MMA_MXF4NVF4_4X]


@pytest.mark.parametrize("form", FORMS)
@pytest.mark.parametrize("pair", [0, 1])
def test_calibration_runs_and_counts(form, pair):
    nsm = torch.cuda.get_device_properties(0).multi_processor_count
    cyc = torch.full((nsm,), -1, dtype=torch.int64, device="cuda")
    per_mma = []
    for steps in (1024, 4096):
        cyc.fill_(-1)
        flops, units = mx.mx_calibrate_mma(form, pair, steps, cyc)
        torch.cuda.synchronize()
        assert mx.mx_device_status() == mx.MX_OK
        assert 1 <= units <= (nsm // 2 if pair else nsm)
        m = 256 if pair else 128
        assert flops == units * steps * 4 * 2 * m * 256 * 64
        c = cyc[:units].cpu()
        assert bool((c > 0).all()), "a unit did not report its cycles"
        assert bool((cyc[units:].cpu() == -1).all()), "wrote past the units it ran"
        per_mma.append(float(c.double().median()) / (4 * steps))
    # a rate: the cost per MMA does not shrink with more MMAs beyond start-up noise,
    # and lies in a plausible range for one 128 x 256 x 64 FP4 MMA per SM
    assert 32 <= per_mma[1] <= 1024
    assert abs(per_mma[1] - per_mma[0]) <= 0.05 * per_mma[1] + 8


def test_calibration_rejects_a_short_cycles_buffer():
    cyc = torch.zeros(4, dtype=torch.int64, device="cuda")
    with pytest.raises(mx.MXError) as e:
        mx.mx_calibrate_mma(mx.MX_MMA_MXF4, 1, 16, cyc)
    assert e.value.code == mx.MX_ERR_INVALID_ARG
    assert "cycles_capacity = 4" in e.value.detail
