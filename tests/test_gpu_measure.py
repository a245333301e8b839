"""The exp2-rate measurement behind the bench's secondary ceiling (GPU)."""
import pytest
import torch

import masked_attention_bound_gb300 as fm

pytestmark = pytest.mark.gpu


def test_exp2_rate_is_plausible_and_repeatable():
    """ex2.approx throughput of the whole GPU: between 16 and 64 evaluations
    per clock per SM at 1-2.1 GHz on 100-200 SMs, and two measurements agree
    within 20 %."""
    r1 = fm.measure_exp2_rate()
    r2 = fm.measure_exp2_rate()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    lo, hi = 16 * sms * 1.0e9, 64 * sms * 2.1e9
    assert lo < r1 < hi and lo < r2 < hi, (r1, r2)
    assert abs(r1 - r2) < 0.2 * max(r1, r2)
