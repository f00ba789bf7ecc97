"""Randomised shapes against the float64 oracle.

A fixed-seed draw of sizes, head groupings, page sizes and mask modes for the
dense prefill (bf16 and FP8), prefill chunks over a paged cache (both the
paged kernel and the prefill kernel's ragged mode, chosen by the longest
chunk), packed variable-length batches, decode over a paged cache
(multi-head and grouped) and the backward pass.  The draws mix tile-aligned and ragged lengths, tiny
and multi-tile sequences, and requests with no new tokens, so combinations
that the hand-picked cases do not list still meet the oracle.
"""
import numpy as np
import pytest
import torch

import attention_attn_fwd_03_gb300 as attn
import oracle
from attention_attn_fwd_03_gb300 import inputs

from _parity import TOL_LSE, TOL_O_BF16, TOL_O_FP8, compare, compare_grad, default_scale

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    attn.lib()


def _draw(kind, n, seed):
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        if kind == "dense":
            out.append(dict(B=int(rng.integers(1, 4)), H=int(rng.integers(1, 5)), Nq=int(rng.integers(1, 700)),
                            Nk=int(rng.integers(1, 900)), d=int(rng.choice([64, 128])),
                            causal=bool(rng.integers(0, 2))))
        else:
            H_kv = int(rng.choice([1, 2, 4]))
            G = int(rng.choice([1, 2, 4, 8]))
            q_hi = int(rng.choice([40, 200, 600]))
            out.append(dict(B=int(rng.integers(1, 5)), H=H_kv * G, H_kv=H_kv, d=int(rng.choice([64, 128])),
                            page=int(rng.choice([8, 16, 32, 64, 128, 256])), q_lo=int(rng.integers(0, q_hi // 2 + 1)),
                            q_hi=q_hi, ctx_hi=int(rng.choice([0, 300, 1500])), causal=bool(rng.integers(0, 2))))
    return out


DENSE = _draw("dense", 24, 2024)


def _draw_long(n, seed):
    """Shapes whose units average 48+ key blocks: the decoupled prefill kernel."""
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        causal = bool(rng.integers(0, 2))
        Nk = int(rng.integers(6200, 9000)) if not causal else int(rng.integers(12400, 16000))
        Nq = int(rng.integers(1, 900)) if rng.integers(0, 2) else Nk - int(rng.integers(0, 300))
        out.append(dict(B=1, H=int(rng.integers(1, 3)), Nq=Nq, Nk=Nk, d=int(rng.choice([64, 128])), causal=causal))
    return out


LONG = _draw_long(6, 77)
CHUNKS = _draw("chunks", 24, 7)
VARLEN = _draw("varlen", 16, 99)
FP8 = [dict(c, d=128) for c in _draw("dense", 8, 5)]


def _draw_decode(n, seed):
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        H_kv = int(rng.choice([1, 2, 4, 8]))
        out.append(dict(B=int(rng.integers(1, 9)), H_kv=H_kv, G=int(rng.choice([1, 2, 4, 8, 16])),
                        d=int(rng.choice([64, 128])), page=int(rng.choice([8, 16, 32, 64, 128, 256])),
                        lo=int(rng.integers(0, 200)), hi=int(rng.choice([300, 2000, 5000]))))
    return out


DECODE = _draw_decode(16, 11)
BWD = [dict(c, Nq=min(c["Nq"], 400), Nk=min(c["Nk"], 500)) for c in _draw("dense", 8, 31)]


@pytest.mark.parametrize("i", range(len(DENSE)))
def test_fuzz_dense(i):
    c = DENSE[i]
    q, k, v = inputs.dense_qkv(c["B"], c["H"], c["Nq"], c["Nk"], c["d"], seed=1000 + i)
    scale = default_scale(c["d"])
    o, lse = attn.fwd(q.to(DEV), k.to(DEV), v.to(DEV), causal=c["causal"], scale=scale)
    attn.device_status()
    o_ref, l_ref = oracle.attention(q, k, v, scale, causal=c["causal"])
    compare("fuzz_dense_%d_%s" % (i, c), o, lse, o_ref, l_ref, TOL_O_BF16, TOL_LSE)


@pytest.mark.parametrize("i", range(len(LONG)))
def test_fuzz_dense_long_rows(i):
    c = LONG[i]
    q, k, v = inputs.dense_qkv(c["B"], c["H"], c["Nq"], c["Nk"], c["d"], seed=1500 + i)
    scale = default_scale(c["d"])
    o, lse = attn.fwd(q.to(DEV), k.to(DEV), v.to(DEV), causal=c["causal"], scale=scale)
    attn.device_status()
    o_ref, l_ref = oracle.attention(q, k, v, scale, causal=c["causal"])
    compare("fuzz_dense_long_%d_%s" % (i, c), o, lse, o_ref, l_ref, TOL_O_BF16, TOL_LSE)


@pytest.mark.parametrize("i", range(len(CHUNKS)))
def test_fuzz_chunks(i):
    c = CHUNKS[i]
    max_pages = (c["q_hi"] + c["ctx_hi"]) // c["page"] + 2
    p = inputs.paged_chunks(B=c["B"], H=c["H"], H_kv=c["H_kv"], d=c["d"], page_size=c["page"], max_pages=max_pages,
                            num_pages=c["B"] * max_pages + 5, q_lo=c["q_lo"], q_hi=c["q_hi"], ctx_lo=0,
                            ctx_hi=c["ctx_hi"], seed=2000 + i)
    g = {k: (v.to(DEV) if isinstance(v, torch.Tensor) and k not in ("used_pages", "q_lens") else v)
         for k, v in p.items()}
    scale = default_scale(c["d"])
    o, lse = attn.paged_fwd(g["q"], g["k_cache"], g["v_cache"], g["block_table"], g["seq_lens"],
                            cu_seqlens_q=g["cu_seqlens_q"], max_q_len=max(1, g["max_q_len"]), causal=c["causal"],
                            scale=scale)
    attn.device_status()
    o_ref, l_ref = oracle.paged_attention(p["q"], p["k_cache"], p["v_cache"], p["block_table"], p["seq_lens"], scale,
                                          cu_seqlens_q=p["cu_seqlens_q"], causal=c["causal"])
    compare("fuzz_chunks_%d_%s" % (i, c), o, lse, o_ref, l_ref, TOL_O_BF16, TOL_LSE)


@pytest.mark.parametrize("i", range(len(VARLEN)))
def test_fuzz_varlen(i):
    c = VARLEN[i]
    p = inputs.varlen_qkv(B=c["B"], H=c["H"], H_kv=c["H_kv"], d=c["d"], q_lo=c["q_lo"], q_hi=c["q_hi"], ctx_lo=0,
                          ctx_hi=c["ctx_hi"], seed=3000 + i)
    scale = default_scale(c["d"])
    dv = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in p.items()}
    o, lse = attn.varlen_fwd(dv["q"], dv["k"], dv["v"], dv["cu_seqlens_q"], dv["cu_seqlens_k"],
                             max_q_len=max(1, p["max_q_len"]), max_k_len=max(1, p["max_k_len"]), causal=c["causal"],
                             scale=scale)
    attn.device_status()
    o_ref, l_ref = oracle.varlen_attention(p["q"], p["k"], p["v"], p["cu_seqlens_q"], p["cu_seqlens_k"], scale,
                                           causal=c["causal"])
    compare("fuzz_varlen_%d_%s" % (i, c), o, lse, o_ref, l_ref, TOL_O_BF16, TOL_LSE)


@pytest.mark.parametrize("i", range(len(FP8)))
def test_fuzz_fp8(i):
    c = FP8[i]
    q, k, v = inputs.dense_qkv(c["B"], c["H"], c["Nq"], c["Nk"], 128, seed=4000 + i)
    (q8, dq), (k8, dk), (v8, dv) = (inputs.fp8_quantize(t) for t in (q, k, v))
    scale = default_scale(128)
    o, lse = attn.fwd_fp8(q8.to(DEV), k8.to(DEV), v8.to(DEV), (dq, dk, dv), causal=c["causal"], scale=scale)
    attn.device_status()
    o_ref, l_ref = oracle.attention(q8, k8, v8, scale, causal=c["causal"], descales=(dq, dk, dv))
    compare("fuzz_fp8_%d_%s" % (i, c), o, lse, o_ref, l_ref, TOL_O_FP8, TOL_LSE)


@pytest.mark.parametrize("i", range(len(DECODE)))
def test_fuzz_decode(i):
    """G = 1 runs through both decode entry points (the CUDA-core split kernel and the tensor-core
    paged kernel); G > 1 through the paged kernel."""
    c = DECODE[i]
    H = c["H_kv"] * c["G"]
    max_pages = c["hi"] // c["page"] + 1
    p = inputs.paged_kv(B=c["B"], H=H, d=c["d"], page_size=c["page"], max_pages=max_pages,
                        num_pages=c["B"] * max_pages + 3, len_lo=c["lo"], len_hi=c["hi"], seed=5000 + i,
                        H_kv=c["H_kv"])
    g = {k: (v.to(DEV) if isinstance(v, torch.Tensor) and k != "used_pages" else v) for k, v in p.items()}
    scale = default_scale(c["d"])
    o_ref, l_ref = oracle.paged_attention(p["q"], p["k_cache"], p["v_cache"], p["block_table"], p["seq_lens"], scale)
    o, lse = attn.paged_fwd(g["q"], g["k_cache"], g["v_cache"], g["block_table"], g["seq_lens"], scale=scale)
    attn.device_status()
    compare("fuzz_decode_tc_%d_%s" % (i, c), o, lse, o_ref, l_ref, TOL_O_BF16, TOL_LSE)
    if c["G"] == 1:
        o2, lse2 = attn.paged_decode(g["q"], g["k_cache"], g["v_cache"], g["block_table"], g["seq_lens"], scale=scale)
        attn.device_status()
        compare("fuzz_decode_mha_%d_%s" % (i, c), o2, lse2, o_ref, l_ref, TOL_O_BF16, TOL_LSE)


@pytest.mark.parametrize("i", range(len(BWD)))
def test_fuzz_bwd(i):
    c = BWD[i]
    q, k, v = inputs.dense_qkv(c["B"], c["H"], c["Nq"], c["Nk"], c["d"], seed=6000 + i)
    do = torch.randn((c["B"], c["H"], c["Nq"], c["d"]), generator=torch.Generator().manual_seed(7000 + i),
                     dtype=torch.float32).to(torch.bfloat16)
    scale = default_scale(c["d"])
    qg, kg, vg, dog = (t.to(DEV) for t in (q, k, v, do))
    o, lse = attn.fwd(qg, kg, vg, causal=c["causal"], scale=scale)
    dq, dk, dv = attn.bwd(qg, kg, vg, o, lse, dog, causal=c["causal"], scale=scale)
    attn.device_status()
    ref = oracle.attention_bwd(q, k, v, do, scale, causal=c["causal"])
    for tag, g, r in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
        compare_grad("fuzz_bwd_%d_%s_%s" % (i, c, tag), g, r)
