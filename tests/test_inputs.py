"""The seeded input recipes: reproducible, shaped as documented, FP8 scaling sane."""
import math

import numpy as np
import torch

from attention_attn_fwd_03_gb300 import inputs


def test_dense_inputs_are_seeded_and_ordered():
    q1, k1, v1 = inputs.dense_qkv(1, 2, 5, 7, 8, seed=0)
    q2, k2, v2 = inputs.dense_qkv(1, 2, 5, 7, 8, seed=0)
    assert torch.equal(q1, q2) and torch.equal(k1, k2) and torch.equal(v1, v2)
    g = torch.Generator().manual_seed(0)
    q3 = torch.randn((1, 2, 5, 8), generator=g).to(torch.bfloat16)
    assert torch.equal(q1, q3)  # Q is drawn first
    assert q1.dtype == torch.bfloat16 and k1.shape == (1, 2, 7, 8)


def test_fp8_quantisation_round_trip():
    """e4m3fn keeps 3 mantissa bits: after per-tensor scaling every value's
    round trip is within half a unit in the last place (2^-4 relative for
    normals, 2^-10 absolute in the subnormal range)."""
    x = torch.randn(4, 3, 64, 16, generator=torch.Generator().manual_seed(1)).to(torch.bfloat16)
    x8, ds = inputs.fp8_quantize(x)
    assert x8.dtype == torch.float8_e4m3fn
    s = 1.0 / ds
    assert abs(float(x.abs().max()) * s - 448.0) < 1e-3
    y = x.double() * s
    back = x8.double()
    err = (back - y).abs()
    bound = torch.maximum(y.abs() * 2.0 ** -4, torch.full_like(y, 2.0 ** -10))
    assert bool((err <= bound * (1 + 1e-9)).all())
    z, dz = inputs.fp8_quantize(torch.zeros(3, dtype=torch.bfloat16))
    assert dz == 1.0 and bool((z.float() == 0).all())


def test_paged_inputs_structure():
    p = inputs.paged_kv(B=6, H=2, d=8, page_size=4, max_pages=5, num_pages=40, len_lo=3, len_hi=20, seed=3)
    bt, sl, kc = p["block_table"], p["seq_lens"], p["k_cache"]
    assert bt.shape == (6, 5) and sl.shape == (6,) and kc.shape == (40, 4, 2, 8)
    seen = []
    for r in range(6):
        n = math.ceil(int(sl[r]) / 4)
        assert 3 <= int(sl[r]) <= 20
        assert bool((bt[r, :n] >= 0).all()) and bool((bt[r, n:] == -1).all())
        seen += bt[r, :n].tolist()
    assert len(seen) == len(set(seen))  # no page is shared
    unused = sorted(set(range(40)) - set(seen))
    assert bool(torch.isnan(kc[unused].float()).all())
    assert bool(torch.isfinite(kc[seen].float()).all())


def test_sample_rows_cover_tile_edges():
    rows = inputs.sample_rows(BH=3, Nq=1000, n_random=50, tile=128, seed=0)
    assert np.all(np.diff(rows) > 0) and rows.min() >= 0 and rows.max() < 3000
    for h in range(3):
        for i in (0, 127, 128, 255, 256, 999, 872):
            assert h * 1000 + i in set(rows.tolist())


def test_paged_chunk_inputs_structure():
    p = inputs.paged_chunks(B=5, H=6, H_kv=2, d=8, page_size=4, max_pages=12, num_pages=60, q_lo=0, q_hi=9,
                            ctx_lo=0, ctx_hi=30, seed=4)
    cu, ql, sl, bt, kc, q = p["cu_seqlens_q"], p["q_lens"], p["seq_lens"], p["block_table"], p["k_cache"], p["q"]
    assert cu.shape == (6,) and int(cu[0]) == 0 and torch.equal(cu[1:] - cu[:-1], ql.to(torch.int32))
    assert q.shape == (int(cu[-1]), 6, 8) and kc.shape == (60, 4, 2, 8)
    assert bool((sl >= ql.to(torch.int32)).all()) and int(sl.max()) <= 12 * 4
    assert p["max_q_len"] == int(ql.max())
    seen = []
    for r in range(5):
        n = math.ceil(int(sl[r]) / 4)
        assert bool((bt[r, :n] >= 0).all()) and bool((bt[r, n:] == -1).all())
        seen += bt[r, :n].tolist()
    assert len(seen) == len(set(seen))
    again = inputs.paged_chunks(B=5, H=6, H_kv=2, d=8, page_size=4, max_pages=12, num_pages=60, q_lo=0, q_hi=9,
                                ctx_lo=0, ctx_hi=30, seed=4)
    assert torch.equal(again["q"], q) and torch.equal(again["block_table"], bt)


def test_grouped_cache_keeps_the_draw_order():
    """Grouped KV heads change only the cache shape: table, lengths and q are
    the multi-head recipe's."""
    a = inputs.paged_kv(B=3, H=4, d=8, page_size=4, max_pages=4, num_pages=16, len_lo=1, len_hi=16, seed=5)
    b = inputs.paged_kv(B=3, H=4, d=8, page_size=4, max_pages=4, num_pages=16, len_lo=1, len_hi=16, seed=5,
                        H_kv=2)
    assert torch.equal(a["q"], b["q"]) and torch.equal(a["block_table"], b["block_table"])
    assert b["k_cache"].shape == (16, 4, 2, 8)


def test_varlen_inputs_structure():
    p = inputs.varlen_qkv(B=6, H=4, H_kv=2, d=8, q_lo=0, q_hi=7, ctx_lo=1, ctx_hi=5, seed=6)
    cu_q, cu_k = p["cu_seqlens_q"], p["cu_seqlens_k"]
    assert cu_q.shape == (7,) and cu_k.shape == (7,) and int(cu_q[0]) == 0 and int(cu_k[0]) == 0
    ql, kl = cu_q[1:] - cu_q[:-1], cu_k[1:] - cu_k[:-1]
    assert bool((kl - ql >= 1).all()) and bool((kl - ql <= 5).all())
    assert p["q"].shape == (int(cu_q[-1]), 4, 8) and p["k"].shape == (int(cu_k[-1]), 2, 8)
    assert p["max_q_len"] == int(ql.max()) and p["max_k_len"] == int(kl.max())
