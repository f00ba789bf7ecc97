"""Tensor-core paged attention (attn_paged_fwd) parity against the float64 oracle.

Grouped-query decode (one token per request; G = H / H_kv query heads share a
KV head, from multi-head G = 1 to multi-query G = 128), the serving workload
with 8 KV heads in full, every supported page size (8 .. 1024), head counts
whose group does not divide 128, zero-length requests, prefill chunks appended
to cached prefixes (several query tiles per request, causal and not, requests
with no new tokens, more new tokens than keys, split key ranges merged
across CTAs), bit-identical results under another physical page placement,
and the device-data checks on both paths; the benchmark's chunk workload in its
launch configuration on sampled rows.  Chunks of 128 tokens or more run on the prefill
kernel's ragged mode (two 128-token tiles of one query head per unit, keys
gathered through the block table); shorter ones on the paged kernel.
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
    return {k: (v.to(DEV) if isinstance(v, torch.Tensor) and k not in ("used_pages", "q_lens") else v)
            for k, v in p.items()}


def _run(g, scale, causal=False, chunks=False):
    o, lse = attn.paged_fwd(g["q"], g["k_cache"], g["v_cache"], g["block_table"], g["seq_lens"],
                            cu_seqlens_q=g["cu_seqlens_q"] if chunks else None,
                            max_q_len=g["max_q_len"] if chunks else None, causal=causal, scale=scale)
    attn.device_status()
    return o, lse


def _ref(p, scale, causal=False, chunks=False):
    return oracle.paged_attention(p["q"].cpu(), p["k_cache"].cpu(), p["v_cache"].cpu(), p["block_table"].cpu(),
                                  p["seq_lens"].cpu(), scale,
                                  cu_seqlens_q=p["cu_seqlens_q"].cpu() if chunks else None, causal=causal)


@pytest.mark.parametrize("B,H,H_kv,d,page,max_pages,lo,hi", [
    (5, 8, 2, 128, 16, 9, 0, 144),        # zero-length requests possible
    (7, 4, 1, 64, 64, 4, 1, 256),         # multi-query, d = 64
    (3, 32, 8, 128, 64, 130, 8000, 8320),  # long: many splits
    (4, 6, 3, 64, 8, 40, 300, 320),       # 8-token pages: 16 boxes per key block
    (2, 32, 4, 128, 128, 3, 384, 384),    # exact page multiples
    (3, 16, 2, 128, 256, 5, 1, 1280),     # pages longer than a key block
    (2, 24, 8, 128, 1024, 2, 1, 2048),    # G = 3: 126 of 128 tile rows used
    (2, 128, 1, 128, 64, 4, 1, 256),      # G = 128: the whole tile is one token
    (3, 4, 4, 128, 32, 8, 1, 256),        # G = 1 (multi-head)
    (12, 32, 8, 128, 64, 100, 1, 6000),   # lengths 1..6000: short requests run unsplit, long ones split
    (40, 16, 4, 64, 16, 300, 0, 4800),    # many streams, empty requests possible
])
def test_grouped_decode(B, H, H_kv, d, page, max_pages, lo, hi):
    p = inputs.paged_kv(B=B, H=H, d=d, page_size=page, max_pages=max_pages, num_pages=B * max_pages + 7,
                        len_lo=lo, len_hi=hi, seed=B + H + d + page, H_kv=H_kv)
    scale = default_scale(d)
    o, lse = _run(_gpu(p), scale)
    o_ref, l_ref = _ref(p, scale)
    compare("gqa_decode_%dx%d/%d_d%d_p%d" % (B, H, H_kv, d, page), o, lse, o_ref, l_ref, TOL_O_BF16, TOL_LSE)


def test_grouped_decode_workload_full():
    """64 requests, 32 query heads over 8 KV heads, d = 128, 64-token pages,
    lengths uniform in [512, 8192], 8192-page pool: every output checked."""
    p = inputs.paged_kv(B=64, H=32, d=128, page_size=64, max_pages=128, num_pages=8192, len_lo=512,
                        len_hi=8192, seed=0, device=DEV, H_kv=8)
    scale = default_scale(128)
    o, lse = _run(p, scale)
    o_ref, l_ref = _ref(p, scale)
    compare("gqa_decode_workload", o, lse, o_ref, l_ref, TOL_O_BF16, TOL_LSE)


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("B,H,H_kv,d,page,max_pages,q_lo,q_hi,ctx_lo,ctx_hi", [
    (4, 8, 2, 128, 64, 16, 1, 300, 0, 700),     # 32 tokens x 4 heads per tile
    (3, 4, 4, 64, 16, 40, 0, 400, 0, 200),      # 128 tokens per tile; empty requests possible
    (2, 12, 3, 128, 32, 64, 500, 900, 100, 1000),
    (1, 8, 8, 128, 64, 100, 150, 250, 5500, 6000),  # few units: split key ranges over several tiles
    (3, 8, 2, 128, 64, 16, 1, 100, 0, 700),     # chunks under 128 tokens: the paged kernel's packed tiles
    (2, 8, 2, 64, 8, 120, 130, 300, 0, 600),    # 8-token pages: 16 boxes per key block, d = 64
    (2, 8, 2, 128, 16, 170, 128, 400, 1500, 2300),  # 16-token pages, d = 128: rows staged 4 blocks at a time
    (2, 4, 1, 128, 256, 6, 200, 400, 100, 1000),  # pages longer than a key block
])
def test_prefill_chunks(B, H, H_kv, d, page, max_pages, q_lo, q_hi, ctx_lo, ctx_hi, causal):
    p = inputs.paged_chunks(B=B, H=H, H_kv=H_kv, d=d, page_size=page, max_pages=max_pages,
                            num_pages=B * max_pages + 5, q_lo=q_lo, q_hi=q_hi, ctx_lo=ctx_lo, ctx_hi=ctx_hi,
                            seed=B * 7 + H + page)
    scale = default_scale(d)
    o, lse = _run(_gpu(p), scale, causal=causal, chunks=True)
    o_ref, l_ref = _ref(p, scale, causal=causal, chunks=True)
    compare("chunks_%dx%d/%d_d%d_p%d_%s" % (B, H, H_kv, d, page, "causal" if causal else "full"), o, lse,
            o_ref, l_ref, TOL_O_BF16, TOL_LSE)


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("B,H,H_kv,d,page,max_pages,q_lo,q_hi,ctx_lo,ctx_hi", [
    (3, 8, 2, 128, 64, 100, 1, 300, 4000, 6000),    # long prefixes
    (4, 8, 2, 64, 16, 400, 0, 260, 0, 6000),        # d = 64; short, long and empty requests
    (3, 4, 4, 128, 8, 800, 128, 400, 5000, 6000),   # 8-token pages: 16 boxes per key block
    (3, 16, 2, 128, 256, 25, 1, 200, 0, 6000),      # pages longer than a key block
    (6, 4, 1, 128, 128, 48, 1, 130, 0, 120),        # short requests only: one key block per unit
])
def test_prefill_chunks_long_key_capacity(B, H, H_kv, d, page, max_pages, q_lo, q_hi, ctx_lo, ctx_hi, causal):
    """Block tables of 6144 keys or more: long prefixes beside short and empty requests and units of
    one key block, with the NaN-filled rest of every partial page past a sequence's end."""
    p = inputs.paged_chunks(B=B, H=H, H_kv=H_kv, d=d, page_size=page, max_pages=max_pages,
                            num_pages=B * max_pages + 5, q_lo=q_lo, q_hi=q_hi, ctx_lo=ctx_lo, ctx_hi=ctx_hi,
                            seed=B * 11 + H + page)
    scale = default_scale(d)
    o, lse = _run(_gpu(p), scale, causal=causal, chunks=True)
    o_ref, l_ref = _ref(p, scale, causal=causal, chunks=True)
    compare("chunks_long_%dx%d/%d_d%d_p%d_%s" % (B, H, H_kv, d, page, "causal" if causal else "full"), o, lse,
            o_ref, l_ref, TOL_O_BF16, TOL_LSE)


@pytest.mark.parametrize("max_pages", [8, 100])
def test_prefill_chunk_longer_than_its_keys(max_pages):
    """seq_len < q_len: under the causal mask the first q_len - seq_len
    queries see no key (O = 0, LSE = -inf); the rest see a prefix."""
    p = inputs.paged_chunks(B=3, H=4, H_kv=2, d=128, page_size=64, max_pages=max_pages, num_pages=3 * max_pages + 16,
                            q_lo=200, q_hi=260, ctx_lo=0, ctx_hi=100, seed=31)
    p["seq_lens"] = (p["seq_lens"] - torch.tensor([150, 0, 230], dtype=torch.int32)).clamp(min=0)
    scale = default_scale(128)
    o, lse = _run(_gpu(p), scale, causal=True, chunks=True)
    o_ref, l_ref = _ref(p, scale, causal=True, chunks=True)
    assert np.isneginf(l_ref).any()
    compare("chunks_short_keys", o, lse, o_ref, l_ref, TOL_O_BF16, TOL_LSE)


@pytest.mark.parametrize("max_pages,q_lo,q_hi", [(12, 1, 100), (200, 130, 300)])
def test_placement_invariance(max_pages, q_lo, q_hi):
    """Moving pages to other physical slots (and the table with them) gives bit-identical output."""
    n = 3 * max_pages + 4
    p = _gpu(inputs.paged_chunks(B=3, H=8, H_kv=2, d=128, page_size=32, max_pages=max_pages, num_pages=n, q_lo=q_lo,
                                 q_hi=q_hi, ctx_lo=0, ctx_hi=280, seed=23))
    o1, l1 = _run(p, default_scale(128), causal=True, chunks=True)
    perm = torch.randperm(n, generator=torch.Generator().manual_seed(4)).to(DEV)
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(n, device=DEV)
    bt = p["block_table"]
    bt2 = torch.where(bt >= 0, inv[bt.clamp(min=0).long()].to(torch.int32), bt)
    p2 = dict(p, k_cache=p["k_cache"][perm].contiguous(), v_cache=p["v_cache"][perm].contiguous(),
              block_table=bt2.contiguous())
    o2, l2 = _run(p2, default_scale(128), causal=True, chunks=True)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_bad_device_data_is_reported():
    p = _gpu(inputs.paged_kv(B=3, H=8, d=128, page_size=16, max_pages=4, num_pages=20, len_lo=20, len_hi=64,
                             seed=24, H_kv=2))
    sl = p["seq_lens"].clone()
    sl[1] = 10_000  # past max_pages * page_size: clamped, reported
    bt = p["block_table"].clone()
    bt[1] = torch.tensor([0, 1, 2, 3], dtype=torch.int32, device=DEV)
    o, _ = attn.paged_fwd(p["q"], p["k_cache"], p["v_cache"], bt, sl)
    with pytest.raises(attn.AttnError) as ei:
        attn.device_status()
    assert ei.value.status == attn.ATTN_ERR_DEVICE_DATA
    bt = p["block_table"].clone()
    bt[0, 0] = 20  # one past the pool: read as zeros, reported
    attn.paged_fwd(p["q"], p["k_cache"], p["v_cache"], bt, p["seq_lens"])
    with pytest.raises(attn.AttnError) as ei:
        attn.device_status()
    assert ei.value.status == attn.ATTN_ERR_DEVICE_DATA
    attn.device_status()  # cleared by the read above
    o, lse = _run(p, default_scale(128))
    o_ref, l_ref = _ref(p, default_scale(128))
    compare("gqa_after_error", o, lse, o_ref, l_ref, TOL_O_BF16, TOL_LSE)


@pytest.mark.parametrize("max_pages", [20, 200])
def test_bad_device_data_is_reported_for_long_chunks(max_pages):
    """The same device-data checks on the ragged path (chunks of 128 tokens or more; both prefill kernels)."""
    p = _gpu(inputs.paged_chunks(B=3, H=8, H_kv=2, d=128, page_size=32, max_pages=max_pages, num_pages=3 * max_pages + 10,
                                 q_lo=130, q_hi=200, ctx_lo=0, ctx_hi=300, seed=41))
    sl = p["seq_lens"].clone()
    sl[1] = 100_000  # past max_pages * page_size: clamped, reported
    attn.paged_fwd(p["q"], p["k_cache"], p["v_cache"], p["block_table"], sl, cu_seqlens_q=p["cu_seqlens_q"],
                   max_q_len=p["max_q_len"], causal=True)
    with pytest.raises(attn.AttnError) as ei:
        attn.device_status()
    assert ei.value.status == attn.ATTN_ERR_DEVICE_DATA
    bt = p["block_table"].clone()
    bt[0, 0] = 3 * max_pages + 10  # one past the pool: read as zeros, reported
    attn.paged_fwd(p["q"], p["k_cache"], p["v_cache"], bt, p["seq_lens"], cu_seqlens_q=p["cu_seqlens_q"],
                   max_q_len=p["max_q_len"], causal=True)
    with pytest.raises(attn.AttnError) as ei:
        attn.device_status()
    assert ei.value.status == attn.ATTN_ERR_DEVICE_DATA
    o, lse = _run(p, default_scale(128), causal=True, chunks=True)
    o_ref, l_ref = _ref(p, default_scale(128), causal=True, chunks=True)
    compare("ragged_after_error", o, lse, o_ref, l_ref, TOL_O_BF16, TOL_LSE)


def _sample(H, q_len, seed, n_random=512):
    """Flattened (head * q_len + token) rows: the first, boundary and last rows of every head, plus random ones."""
    g = torch.Generator().manual_seed(seed)
    per = sorted({0, 1, 127, 128, 255, 256, q_len // 2, q_len - 2, q_len - 1} & set(range(q_len)))
    rows = {h * q_len + i for h in range(H) for i in per}
    rows |= set(torch.randint(0, H * q_len, (n_random,), generator=g).tolist())
    return np.array(sorted(rows), dtype=np.int64)


def _check_sampled(name, o, lse, q, k_rows, v_rows, q_start, q_len, H, H_kv, scale, seed):
    """Oracle on sampled rows of one request: dense [1, H, L, d] keys expanded over the G heads of a KV head."""
    G = H // H_kv
    qd = q[q_start:q_start + q_len].permute(1, 0, 2).unsqueeze(0).contiguous()
    kd = k_rows.permute(1, 0, 2).repeat_interleave(G, dim=0).unsqueeze(0).contiguous()
    vd = v_rows.permute(1, 0, 2).repeat_interleave(G, dim=0).unsqueeze(0).contiguous()
    rows = _sample(H, q_len, seed)
    o_ref, l_ref = oracle.attention(qd, kd, vd, scale, causal=True, rows=rows)
    hh, tt = torch.from_numpy(rows // q_len), torch.from_numpy(rows % q_len)
    o_sel = o.cpu()[q_start + tt, hh]
    l_sel = lse.cpu()[q_start + tt, hh]
    compare(name, o_sel, l_sel, o_ref, l_ref, TOL_O_BF16, TOL_LSE)


def test_prefill_chunks_workload_sampled():
    """The benchmark's chunk workload in its launch configuration (8 requests x 2048 new tokens after 6144
    cached, 32 query heads over 8 KV heads, d = 128, 64-token pages): sampled rows of every request."""
    p = inputs.paged_chunks(B=8, H=32, H_kv=8, d=128, page_size=64, max_pages=128, num_pages=1024, q_lo=2048,
                            q_hi=2048, ctx_lo=6144, ctx_hi=6144, seed=0, device=DEV)
    scale = default_scale(128)
    o, lse = _run(p, scale, causal=True, chunks=True)
    q, kc, vc = p["q"].cpu(), p["k_cache"].cpu(), p["v_cache"].cpu()
    bt, sl, cu = p["block_table"].cpu(), p["seq_lens"].cpu(), p["cu_seqlens_q"].cpu()
    for r in range(8):
        L = int(sl[r])
        pages = bt[r, :(L + 63) // 64].long()
        k_rows = kc[pages].reshape(-1, 8, 128)[:L]
        v_rows = vc[pages].reshape(-1, 8, 128)[:L]
        _check_sampled("chunks_workload_r%d" % r, o, lse, q, k_rows, v_rows, int(cu[r]), int(cu[r + 1] - cu[r]),
                       32, 8, scale, r)
