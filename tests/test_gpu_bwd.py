"""Backward pass (attn_bwd) parity against the float64 gradient oracle.

The forward kernel supplies O and the LSE; the upstream gradient dO is a
seeded N(0,1) bf16 tensor.  Cases: d = 64 and 128, causal and not, ragged
lengths (tail blocks on both axes, for d = 128 also of its 64-query blocks), Nq != Nk under the bottom-right causal
mask (rows with no visible key, keys no query sees), several heads, and the
batched 4 x 16 x 2048 workload checked on a subset of heads.
"""
import math

import numpy as np
import pytest
import torch

import attention_attn_fwd_03_gb300 as attn
import oracle
from attention_attn_fwd_03_gb300 import inputs

from _parity import compare_grad, default_scale

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    attn.lib()


def _dout(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=g, dtype=torch.float32).to(torch.bfloat16)


def _check(B, H, Nq, Nk, d, causal, seed, heads=None):
    q, k, v = inputs.dense_qkv(B, H, Nq, Nk, d, seed=seed)
    do = _dout((B, H, Nq, d), seed + 1)
    scale = default_scale(d)
    qg, kg, vg, dog = (t.to(DEV) for t in (q, k, v, do))
    o, lse = attn.fwd(qg, kg, vg, causal=causal, scale=scale)
    dq, dk, dv = attn.bwd(qg, kg, vg, o, lse, dog, causal=causal, scale=scale)
    attn.device_status()
    sel = (slice(None), slice(None)) if heads is None else (slice(0, 1), slice(0, heads))
    ref = oracle.attention_bwd(q[sel], k[sel], v[sel], do[sel], scale, causal=causal)
    name = "bwd_%dx%dx%dx%d_d%d_%s" % (B, H, Nq, Nk, d, "causal" if causal else "full")
    for tag, g, r in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
        compare_grad(name + "_" + tag, g[sel], r)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,H,Nq,Nk,d", [
    (1, 2, 256, 256, 128),
    (1, 2, 256, 256, 64),
    (2, 3, 300, 300, 128),   # tail blocks
    (1, 2, 200, 456, 128),   # more keys than queries
    (1, 2, 456, 200, 64),    # more queries than keys: rows with no key under the causal mask
    (1, 2, 456, 200, 128),
    (1, 3, 40, 300, 128),    # fewer queries than one 64-row block (d = 128 runs 64-query blocks)
    (1, 2, 65, 129, 128),    # one query past a 64-row block, one key past a 128-key block
    (2, 4, 1024, 1024, 128),
    (2, 24, 700, 700, 128),  # more (head, key block) units than SMs: causal CTAs loop over units
    (1, 40, 333, 520, 128),
])
def test_bwd(B, H, Nq, Nk, d, causal):
    _check(B, H, Nq, Nk, d, causal, seed=B * 100 + Nq + d)


def test_bwd_batched_workload_sampled_heads():
    """4 x 16 x 2048 x 2048, d = 128, causal: the first four heads checked in full."""
    _check(4, 16, 2048, 2048, 128, True, seed=0, heads=4)
