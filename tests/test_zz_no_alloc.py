"""The allocation-free paged decode entry point, attn_paged_decode_noalloc.

It serves callers that cannot allocate device memory at call time (a serving
loop whose memory is fully reserved for its own KV-cache pool, or one that
forbids cudaMalloc after start-up because it can synchronise the device).
It keeps the split partials in the library's fixed device scratch array, so
this test checks, through the C ABI, that two calls in a row match the float64
oracle within the decode tolerances and the workspace-taking entry point
(bit for bit when both use the same split plan), and that a problem too large
for the fixed array is refused before anything is enqueued.

This file is named so that pytest collects it last.
"""
import numpy as np
import pytest
import torch

import attention_attn_fwd_03_gb300 as attn
import oracle
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
    o_ws, l_ws = attn.paged_decode(p["q"], p["k_cache"], p["v_cache"], p["block_table"], p["seq_lens"],
                                   scale=scale)
    attn.device_status()
    o_ws = o_ws.float().cpu().numpy()
    l_ws = l_ws.cpu().numpy()
    o_ref, l_ref = oracle.paged_decode(p["q"].cpu(), p["k_cache"].cpu(), p["v_cache"].cpu(),
                                       p["block_table"].cpu(), p["seq_lens"].cpu(), scale)
    empty = np.isneginf(l_ref)
    # the fixed scratch holds the default plan's partials for the small case
    # (same split plan, so the same arithmetic in the same order); the serving
    # workload needs a coarser split, which changes only the fp32 rounding
    same_plan = attn.attn_paged_decode_workspace_size(B, H, d, max_pages, page) <= attn.ATTN_NOALLOC_SCRATCH_BYTES
    for _ in range(2):  # two calls in a row share the same scratch array
        o = torch.full_like(p["q"], float("nan"))
        lse = torch.full((B, H), float("nan"), dtype=torch.float32, device=DEV)
        assert _call_noalloc(p, scale, o, lse) == attn.ATTN_OK
        attn.device_status()
        o_np, l_np = o.float().cpu().numpy(), lse.cpu().numpy()
        assert np.all(np.isfinite(o_np))
        assert np.array_equal(np.isneginf(l_np), empty)
        assert np.all(o_np[empty] == 0.0)
        # against the float64 oracle, at the decode tolerances
        assert np.max(np.abs(o_np - o_ref)) <= TOL_O_BF16
        assert np.max(np.abs(l_np[~empty] - l_ref[~empty])) <= TOL_LSE
        # against the workspace entry point
        if same_plan:
            assert np.array_equal(o_np, o_ws) and np.array_equal(l_np, l_ws)
        else:
            assert np.max(np.abs(o_np - o_ws)) <= TOL_O_BF16
            assert np.max(np.abs(l_np[~empty] - l_ws[~empty])) <= TOL_LSE


def test_noalloc_refuses_problems_beyond_the_fixed_scratch():
    """4096 requests x 128 heads need ~272 MB of partials even at one split per
    request: refused with ATTN_ERR_WORKSPACE, nothing enqueued.  Every buffer is
    allocated at the shape passed in, so even a wrongly accepted call would
    stay inside them."""
    attn.lib()
    B, H, d, page, max_pages, num_pages = 4096, 128, 128, 8, 4, 8
    q = torch.zeros((B, H, d), dtype=torch.bfloat16, device=DEV)
    k_cache = torch.zeros((num_pages, page, H, d), dtype=torch.bfloat16, device=DEV)
    v_cache = torch.zeros_like(k_cache)
    block_table = torch.zeros((B, max_pages), dtype=torch.int32, device=DEV)
    seq_lens = torch.ones((B,), dtype=torch.int32, device=DEV)
    o = torch.full((B, H, d), 3.0, dtype=torch.bfloat16, device=DEV)
    lse = torch.full((B, H), 3.0, dtype=torch.float32, device=DEV)
    st = attn.attn_paged_decode_noalloc(
        q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), block_table.data_ptr(), seq_lens.data_ptr(),
        B, H, d, page, max_pages, num_pages, 0.088, o.data_ptr(), lse.data_ptr(),
        torch.cuda.current_stream().cuda_stream)
    assert st == attn.ATTN_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert bool((o == 3.0).all()) and bool((lse == 3.0).all())  # nothing was enqueued
