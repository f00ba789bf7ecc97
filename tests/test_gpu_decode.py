"""Paged-KV decode parity against the float64 oracle.

Covers the serving workload (64 requests, H=32, d=128, 64-token pages, lengths
uniform in [512, 8192], random non-repeating pages from an 8192-page pool,
unused pages NaN-filled) in full, small cases with odd head counts, d=64,
other page sizes, zero and page-multiple lengths, invariance of the result
under a different physical placement of the same pages, and the device-data
checks (a length past the table and an out-of-range page id are reported
through the status word without any out-of-bounds access).
"""
import numpy as np
import pytest
import torch

import attention_attn_fwd_03_gb300 as attn
import oracle
from attention_attn_fwd_03_gb300 import inputs

from _parity import TOL_LSE, TOL_O_BF16, compare, default_scale

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    attn.lib()


def _gpu(p):
    return {k: (v.to(DEV) if isinstance(v, torch.Tensor) and k != "used_pages" else v) for k, v in p.items()}


def _run(g, scale):
    o, lse = attn.paged_decode(g["q"], g["k_cache"], g["v_cache"], g["block_table"], g["seq_lens"], scale=scale)
    attn.device_status()
    return o, lse


def _ref(p, scale):
    return oracle.paged_decode(p["q"].cpu(), p["k_cache"].cpu(), p["v_cache"].cpu(), p["block_table"].cpu(),
                               p["seq_lens"].cpu(), scale)


@pytest.mark.parametrize("B,H,d,page,max_pages,lo,hi", [
    (5, 3, 128, 16, 9, 0, 144),      # odd head count, zero-length requests possible
    (7, 2, 64, 64, 4, 1, 256),
    (3, 8, 128, 64, 130, 8000, 8320),  # long, many splits
    (4, 5, 64, 8, 40, 300, 320),
    (2, 32, 128, 128, 3, 384, 384),   # exact page multiples
])
def test_decode_small(B, H, d, page, max_pages, lo, hi):
    p = inputs.paged_kv(B=B, H=H, d=d, page_size=page, max_pages=max_pages, num_pages=B * max_pages + 7,
                        len_lo=lo, len_hi=hi, seed=B + H + d + page)
    scale = default_scale(d)
    o, lse = _run(_gpu(p), scale)
    o_ref, l_ref = _ref(p, scale)
    compare("decode_%dx%d_d%d_p%d" % (B, H, d, page), o, lse, o_ref, l_ref, TOL_O_BF16, TOL_LSE)


def test_decode_workload_full():
    """64 requests x 32 heads x d=128, 64-token pages, 8192-page pool: every output checked."""
    p = inputs.paged_kv(B=64, H=32, d=128, page_size=64, max_pages=128, num_pages=8192, len_lo=512,
                        len_hi=8192, seed=0, device=DEV)
    scale = default_scale(128)
    o, lse = _run(p, scale)
    o_ref, l_ref = _ref(p, scale)
    compare("decode_workload", o, lse, o_ref, l_ref, TOL_O_BF16, TOL_LSE)


def test_decode_placement_invariance():
    """Moving pages to other physical slots (and the table with them) gives bit-identical output."""
    p = _gpu(inputs.paged_kv(B=6, H=4, d=128, page_size=32, max_pages=10, num_pages=80, len_lo=1, len_hi=320,
                             seed=21))
    o1, l1 = _run(p, default_scale(128))
    perm = torch.randperm(80, generator=torch.Generator().manual_seed(3)).to(DEV)
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(80, device=DEV)
    bt = p["block_table"]
    bt2 = torch.where(bt >= 0, inv[bt.clamp(min=0).long()].to(torch.int32), bt)
    p2 = dict(p, k_cache=p["k_cache"][perm].contiguous(), v_cache=p["v_cache"][perm].contiguous(),
              block_table=bt2.contiguous())
    o2, l2 = _run(p2, default_scale(128))
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_decode_bad_device_data_is_reported():
    p = _gpu(inputs.paged_kv(B=3, H=2, d=128, page_size=16, max_pages=4, num_pages=20, len_lo=20, len_hi=64,
                             seed=22))
    # a length beyond max_pages * page_size: clamped, reported
    sl = p["seq_lens"].clone()
    sl[1] = 10_000
    bt = p["block_table"].clone()
    bt[1] = torch.tensor([0, 1, 2, 3], dtype=torch.int32, device=DEV)
    attn.paged_decode(p["q"], p["k_cache"], p["v_cache"], bt, sl)
    with pytest.raises(attn.AttnError) as ei:
        attn.device_status()
    assert ei.value.status == attn.ATTN_ERR_DEVICE_DATA
    # a page id past the pool: skipped, reported
    bt = p["block_table"].clone()
    bt[0, 0] = 20
    o, _ = attn.paged_decode(p["q"], p["k_cache"], p["v_cache"], bt, p["seq_lens"])
    with pytest.raises(attn.AttnError) as ei:
        attn.device_status()
    assert ei.value.status == attn.ATTN_ERR_DEVICE_DATA
    assert bool(torch.isfinite(o.float()).all())
    attn.device_status()  # cleared by the read above
    # the regular call still works afterwards
    o, lse = _run(p, default_scale(128))
    o_ref, l_ref = _ref(p, default_scale(128))
    compare("decode_after_error", o, lse, o_ref, l_ref, TOL_O_BF16, TOL_LSE)
