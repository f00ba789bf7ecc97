"""Variable-length batch prefill (attn_varlen_fwd) parity against the float64 oracle.

Packed self-attention batches (causal and not), prefixes longer than the new
tokens, grouped KV heads from G = 1 to 8, d = 64 and 128, empty requests,
requests with more queries than keys, one-token queries over long keys, and
key ranges split over several CTAs and merged; the benchmark's workload in its
launch configuration on sampled rows; more sequence groups than the schedule
keeps apart, and more sequences than it groups.  Launches whose longest
request has 128 queries or more run on the prefill kernel's ragged mode
(query tails of any length inside a tile pair); shorter ones on the paged
kernel, and both are covered.
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


def _run(p, scale, causal):
    d = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in p.items()}
    o, lse = attn.varlen_fwd(d["q"], d["k"], d["v"], d["cu_seqlens_q"], d["cu_seqlens_k"], max_q_len=d["max_q_len"],
                             max_k_len=d["max_k_len"], causal=causal, scale=scale)
    attn.device_status()
    return o, lse


def _ref(p, scale, causal):
    return oracle.varlen_attention(p["q"], p["k"], p["v"], p["cu_seqlens_q"], p["cu_seqlens_k"], scale, causal=causal)


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("B,H,H_kv,d,q_lo,q_hi,ctx_lo,ctx_hi", [
    (6, 8, 2, 128, 1, 700, 0, 0),          # packed self-attention
    (4, 4, 4, 64, 0, 300, 0, 200),         # G = 1, d = 64, empty requests possible
    (3, 16, 2, 128, 1000, 1500, 0, 3000),  # G = 8, few units: key ranges split and merged
    (8, 32, 8, 128, 1, 1, 100, 3000),      # one query per request over long keys
    (5, 8, 2, 128, 20, 100, 0, 400),       # short queries: the paged kernel's packed tiles
    (3, 8, 2, 128, 256, 256, 0, 300),      # whole tile pairs, no ragged query tail
    (4, 6, 3, 64, 129, 520, 0, 900),       # tails of 1..127 rows in either tile, d = 64
])
def test_varlen(B, H, H_kv, d, q_lo, q_hi, ctx_lo, ctx_hi, causal):
    p = inputs.varlen_qkv(B=B, H=H, H_kv=H_kv, d=d, q_lo=q_lo, q_hi=q_hi, ctx_lo=ctx_lo, ctx_hi=ctx_hi,
                          seed=B * 31 + H + d)
    scale = default_scale(d)
    o, lse = _run(p, scale, causal)
    o_ref, l_ref = _ref(p, scale, causal)
    compare("varlen_%dx%d/%d_d%d_q%d-%d_ctx%d-%d_%s" % (B, H, H_kv, d, q_lo, q_hi, ctx_lo, ctx_hi,
                                                        "causal" if causal else "full"),
            o, lse, o_ref, l_ref, TOL_O_BF16, TOL_LSE)


def test_varlen_more_queries_than_keys():
    """Under the causal mask the first q_len - k_len queries see no key."""
    p = inputs.varlen_qkv(B=3, H=8, H_kv=4, d=128, q_lo=200, q_hi=300, seed=41)
    cu_q, cu_k = p["cu_seqlens_q"], p["cu_seqlens_k"].clone()
    lens = cu_k[1:] - cu_k[:-1]
    new_lens = torch.tensor([int(lens[0]) // 3, int(lens[1]), 0], dtype=torch.int64)
    keep = torch.cat([torch.arange(int(cu_k[r]), int(cu_k[r]) + int(new_lens[r])) for r in range(3)])
    p["k"], p["v"] = p["k"][keep].contiguous(), p["v"][keep].contiguous()
    p["cu_seqlens_k"] = torch.cat([torch.zeros(1, dtype=torch.int64), torch.cumsum(new_lens, 0)]).to(torch.int32)
    p["max_k_len"] = int(new_lens.max())
    scale = default_scale(128)
    o, lse = _run(p, scale, True)
    o_ref, l_ref = _ref(p, scale, True)
    assert np.isneginf(l_ref).any()
    compare("varlen_short_keys", o, lse, o_ref, l_ref, TOL_O_BF16, TOL_LSE)


def test_varlen_workload_sampled():
    """The benchmark's varlen workload (16 causal sequences of 512..4096 tokens, 32 query heads over 8 KV
    heads, d = 128) in its launch configuration: sampled rows of every sequence against the oracle."""
    p = inputs.varlen_qkv(B=16, H=32, H_kv=8, d=128, q_lo=512, q_hi=4096, seed=0, device=DEV)
    scale = default_scale(128)
    o, lse = attn.varlen_fwd(p["q"], p["k"], p["v"], p["cu_seqlens_q"], p["cu_seqlens_k"], p["max_q_len"],
                             p["max_k_len"], causal=True, scale=scale)
    attn.device_status()
    q, k, v = p["q"].cpu(), p["k"].cpu(), p["v"].cpu()
    cq, ck = p["cu_seqlens_q"].cpu(), p["cu_seqlens_k"].cpu()
    g = torch.Generator().manual_seed(3)
    for r in range(16):
        q_start, q_len = int(cq[r]), int(cq[r + 1] - cq[r])
        k0, k1 = int(ck[r]), int(ck[r + 1])
        G = 4
        qd = q[q_start:q_start + q_len].permute(1, 0, 2).unsqueeze(0).contiguous()
        kd = k[k0:k1].permute(1, 0, 2).repeat_interleave(G, dim=0).unsqueeze(0).contiguous()
        vd = v[k0:k1].permute(1, 0, 2).repeat_interleave(G, dim=0).unsqueeze(0).contiguous()
        per = sorted({0, 1, 127, 128, 255, 256, q_len // 2, q_len - 1} & set(range(q_len)))
        rows = {h * q_len + i for h in range(32) for i in per}
        rows |= set(torch.randint(0, 32 * q_len, (256,), generator=g).tolist())
        rows = np.array(sorted(rows), dtype=np.int64)
        o_ref, l_ref = oracle.attention(qd, kd, vd, scale, causal=True, rows=rows)
        hh, tt = torch.from_numpy(rows // q_len), torch.from_numpy(rows % q_len)
        compare("varlen_workload_s%d" % r, o.cpu()[q_start + tt, hh], lse.cpu()[q_start + tt, hh], o_ref, l_ref,
                TOL_O_BF16, TOL_LSE)


def test_varlen_many_key_groups():
    """The schedule lists sequences in groups of about 32 MB of keys and values (longest first) and puts
    every sequence past the 16th group into the last one: 20 sequences of ~10k keys (~40 MB each, one KV
    head per query head) form more than 16 groups."""
    p = inputs.varlen_qkv(B=20, H=8, H_kv=8, d=128, q_lo=128, q_hi=200, ctx_lo=9000, ctx_hi=11000, seed=47)
    scale = default_scale(128)
    o, lse = _run(p, scale, True)
    o_ref, l_ref = _ref(p, scale, True)
    compare("varlen_many_groups", o, lse, o_ref, l_ref, TOL_O_BF16, TOL_LSE)


def test_varlen_many_sequences_ungrouped():
    """More than 4096 sequences: the schedule keeps a single longest-first list (no sequence groups)."""
    p = inputs.varlen_qkv(B=4100, H=2, H_kv=1, d=64, q_lo=128, q_hi=128, seed=53)
    scale = default_scale(64)
    o, lse = _run(p, scale, True)
    o_ref, l_ref = _ref(p, scale, True)
    compare("varlen_4100_sequences", o, lse, o_ref, l_ref, TOL_O_BF16, TOL_LSE)
