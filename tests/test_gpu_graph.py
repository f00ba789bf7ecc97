"""The entry points under CUDA graph capture.

A serving loop captures its per-step launches once and replays them.  The
library's calls enqueue kernels only (tensor maps are encoded on the host and
passed by value; workspaces are the caller's), so a captured call must
replay to the same bits as the eager call, and a replay after the inputs
change in place must follow the new inputs.
"""
import pytest
import torch

import attention_attn_fwd_03_gb300 as attn
from attention_attn_fwd_03_gb300 import inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _capture(fn):
    fn()  # warm-up: per-device set-up and kernel attributes outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            fn()
    torch.cuda.current_stream().wait_stream(s)
    return g


def test_prefill_replays_bit_identically():
    q, k, v = (t.to(DEV) for t in inputs.dense_qkv(2, 4, 640, 640, 128, seed=21))
    o, l = torch.empty_like(q), torch.empty((2, 4, 640), dtype=torch.float32, device=DEV)
    g = _capture(lambda: attn.fwd(q, k, v, causal=True, out=o, lse=l))
    o_ref, l_ref = attn.fwd(q, k, v, causal=True)
    o.zero_()
    g.replay()
    torch.cuda.synchronize()
    attn.device_status()
    assert torch.equal(o, o_ref) and torch.equal(l, l_ref)
    q2, k2, v2 = (t.to(DEV) for t in inputs.dense_qkv(2, 4, 640, 640, 128, seed=22))
    q.copy_(q2), k.copy_(k2), v.copy_(v2)
    g.replay()
    torch.cuda.synchronize()
    o_ref2, l_ref2 = attn.fwd(q2, k2, v2, causal=True)
    attn.device_status()
    assert torch.equal(o, o_ref2) and torch.equal(l, l_ref2)


def test_long_row_prefill_replays_bit_identically():
    """The decoupled prefill kernel (long rows) under graph capture."""
    q, k, v = (t.to(DEV) for t in inputs.dense_qkv(1, 2, 300, 6400, 128, seed=24))
    o, l = torch.empty_like(q), torch.empty((1, 2, 300), dtype=torch.float32, device=DEV)
    g = _capture(lambda: attn.fwd(q, k, v, causal=True, out=o, lse=l))
    o_ref, l_ref = attn.fwd(q, k, v, causal=True)
    o.zero_()
    g.replay()
    torch.cuda.synchronize()
    attn.device_status()
    assert torch.equal(o, o_ref) and torch.equal(l, l_ref)


def test_paged_decode_and_chunks_replay_bit_identically():
    p = inputs.paged_kv(B=16, H=32, d=128, page_size=64, max_pages=32, num_pages=600, len_lo=100, len_hi=2048,
                        seed=23, device=DEV, H_kv=8)
    ws = torch.empty(attn.attn_paged_fwd_workspace_size(16, 16, 1, 32, 8, 128, 64, 32), dtype=torch.uint8,
                     device=DEV)
    o = torch.empty_like(p["q"])
    l = torch.empty((16, 32), dtype=torch.float32, device=DEV)
    g = _capture(lambda: attn.paged_fwd(p["q"], p["k_cache"], p["v_cache"], p["block_table"], p["seq_lens"],
                                        out=o, lse=l, workspace=ws))
    o_ref, l_ref = attn.paged_fwd(p["q"], p["k_cache"], p["v_cache"], p["block_table"], p["seq_lens"])
    o.zero_()
    g.replay()
    torch.cuda.synchronize()
    attn.device_status()
    assert torch.equal(o, o_ref) and torch.equal(l, l_ref)
    # new lengths in place: the captured schedule pass reads them on every replay
    p["seq_lens"].copy_((p["seq_lens"] // 2).clamp(min=1))
    g.replay()
    torch.cuda.synchronize()
    o_ref2, l_ref2 = attn.paged_fwd(p["q"], p["k_cache"], p["v_cache"], p["block_table"], p["seq_lens"])
    attn.device_status()
    assert torch.equal(o, o_ref2) and torch.equal(l, l_ref2)

    c = inputs.paged_chunks(B=3, H=8, H_kv=2, d=128, page_size=64, max_pages=16, num_pages=60, q_lo=130,
                            q_hi=300, ctx_lo=0, ctx_hi=600, seed=24, device=DEV)
    mq = c["max_q_len"]
    wsc = torch.empty(attn.attn_paged_fwd_workspace_size(3, c["q"].shape[0], mq, 8, 2, 128, 64, 16),
                      dtype=torch.uint8, device=DEV)
    oc = torch.empty_like(c["q"])
    lc = torch.empty((c["q"].shape[0], 8), dtype=torch.float32, device=DEV)
    gc = _capture(lambda: attn.paged_fwd(c["q"], c["k_cache"], c["v_cache"], c["block_table"], c["seq_lens"],
                                         cu_seqlens_q=c["cu_seqlens_q"], max_q_len=mq, causal=True, out=oc,
                                         lse=lc, workspace=wsc))
    oc_ref, lc_ref = attn.paged_fwd(c["q"], c["k_cache"], c["v_cache"], c["block_table"], c["seq_lens"],
                                    cu_seqlens_q=c["cu_seqlens_q"], max_q_len=mq, causal=True)
    oc.zero_()
    gc.replay()
    torch.cuda.synchronize()
    attn.device_status()
    assert torch.equal(oc, oc_ref) and torch.equal(lc, lc_ref)
