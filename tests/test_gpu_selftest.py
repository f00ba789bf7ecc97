"""The tensor-core rate check (attn_selftest_mma_rate) through the C ABI: one
CTA per SM times back-to-back 128x128x16 bf16 tcgen05.mma, the denominator of
the prefill roofline.  Checked for sane, consistent values (every CTA timed,
rates within a factor of two of each other and of one MMA per 64 cycles)."""
import statistics

import pytest
import torch

import attention_attn_fwd_03_gb300 as attn

pytestmark = pytest.mark.gpu
DEV = "cuda"


def test_mma_rate_per_sm():
    attn.lib()
    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    cyc = torch.zeros(n_sm, dtype=torch.int64, device=DEV)
    n_groups = 1024
    st = attn.attn_selftest_mma_rate(cyc.data_ptr(), n_sm, n_groups, torch.cuda.current_stream().cuda_stream)
    assert st == attn.ATTN_OK
    attn.device_status()
    c = cyc.cpu().tolist()
    assert all(x > 0 for x in c)
    rates = [4 * n_groups * 2 * 128 * 128 * 16 / x for x in c]  # FLOP per SM cycle
    med = statistics.median(rates)
    assert 4096 <= med <= 16384, med
    assert all(0.5 * med <= r <= 2.0 * med for r in rates)
