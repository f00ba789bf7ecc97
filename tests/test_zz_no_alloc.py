"""The allocation-free paged decode entry point, attn_paged_decode_noalloc.

It serves callers that cannot allocate device memory at call time (a serving
loop whose memory is fully reserved for its own KV-cache pool, or one that
forbids cudaMalloc after start-up because it can synchronise the device).
It keeps the split partials in the library's fixed device scratch array, so
this test checks, through the C ABI, that two calls in a row match the
workspace-taking entry point within the decode tolerances, and that a problem
too large for the fixed array is refused before anything is enqueued.

This file is named so that pytest collects it last.
"""
import numpy as np
import pytest
import torch

import attention_attn_fwd_03_gb300 as attn
from attention_attn_fwd_03_gb300 import inputs

from _parity import TOL_LSE, TOL_O_BF16, default_scale

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _call_noalloc(p, scale, o, lse):
    B, H, d = p["q"].shape
    num_pages, page = p["k_cache"].shape[0], p["k_cache"].shape[1]
    return attn.attn_paged_decode_noalloc(
        p["q"].data_ptr(), p["k_cache"].data_ptr(), p["v_cache"].data_ptr(), p["block_table"].data_ptr(),
        p["seq_lens"].data_ptr(), B, H, d, page, p["block_table"].shape[1], num_pages, scale, o.data_ptr(),
        lse.data_ptr(), torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("B,H,d,page,max_pages,num_pages,lo,hi", [
    (5, 3, 128, 16, 9, 60, 0, 144),            # small, zero-length requests possible
    (64, 32, 128, 64, 128, 8192, 512, 8192),   # serving workload: needs a coarser split to fit
])
def test_noalloc_matches_workspace_entry_point(B, H, d, page, max_pages, num_pages, lo, hi):
    attn.lib()
    p = inputs.paged_kv(B=B, H=H, d=d, page_size=page, max_pages=max_pages, num_pages=num_pages, len_lo=lo,
                        len_hi=hi, seed=B + H, device=DEV)
    scale = default_scale(d)
    o_ref, l_ref = attn.paged_decode(p["q"], p["k_cache"], p["v_cache"], p["block_table"], p["seq_lens"],
                                     scale=scale)
    attn.device_status()
    o_ref = o_ref.float().cpu().numpy()
    l_ref = l_ref.cpu().numpy()
    empty = np.isneginf(l_ref)
    for _ in range(2):  # two calls in a row share the same scratch array
        o = torch.full_like(p["q"], float("nan"))
        lse = torch.full((B, H), float("nan"), dtype=torch.float32, device=DEV)
        assert _call_noalloc(p, scale, o, lse) == attn.ATTN_OK
        attn.device_status()
        o_np, l_np = o.float().cpu().numpy(), lse.cpu().numpy()
        assert np.all(np.isfinite(o_np))
        assert np.array_equal(np.isneginf(l_np), empty)
        assert np.max(np.abs(o_np - o_ref)) <= TOL_O_BF16
        assert np.max(np.abs(l_np[~empty] - l_ref[~empty])) <= TOL_LSE


def test_noalloc_refuses_problems_beyond_the_fixed_scratch():
    attn.lib()
    p = inputs.paged_kv(B=2, H=2, d=128, page_size=8, max_pages=4, num_pages=8, len_lo=1, len_hi=32, seed=5,
                        device=DEV)
    o = torch.zeros_like(p["q"])
    lse = torch.zeros((2, 2), dtype=torch.float32, device=DEV)
    # one split per request for 4096 requests x 128 heads needs ~272 MB of partials
    st = attn.attn_paged_decode_noalloc(
        p["q"].data_ptr(), p["k_cache"].data_ptr(), p["v_cache"].data_ptr(), p["block_table"].data_ptr(),
        p["seq_lens"].data_ptr(), 4096, 128, 128, 8, 4, 8, 0.088, o.data_ptr(), lse.data_ptr(),
        torch.cuda.current_stream().cuda_stream)
    assert st == attn.ATTN_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert bool((o == 0).all()) and bool((lse == 0).all())  # nothing was enqueued
