"""FP8-e4m3 prefill parity against the float64 oracle run on the dequantised inputs.

Workload: B=2, H=16, N=8192, d=128, non-causal, per-tensor amax scaling,
every output element checked, plus small full checks incl. causal and ragged
shapes.  O tolerance 6e-2; LSE is checked at 1e-3 as well since l is summed
from unquantised probabilities.
"""
import pytest
import torch

import attention_attn_fwd_03_gb300 as attn
import oracle
from attention_attn_fwd_03_gb300 import inputs

from _parity import TOL_LSE, TOL_O_FP8, compare, default_scale

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    attn.lib()


def _quant(q, k, v):
    return inputs.fp8_quantize(q), inputs.fp8_quantize(k), inputs.fp8_quantize(v)


def _run(q8, k8, v8, ds, causal, scale):
    o, lse = attn.fwd_fp8(q8.to(DEV), k8.to(DEV), v8.to(DEV), ds, causal=causal, scale=scale)
    attn.device_status()
    return o, lse


@pytest.mark.parametrize("B,H,Nq,Nk,causal", [(1, 1, 256, 256, False), (1, 2, 300, 300, True),
                                              (2, 1, 129, 1000, False), (1, 1, 1, 1, False),
                                              (1, 1, 700, 5, True), (1, 2, 512, 512, True)])
def test_fp8_small(B, H, Nq, Nk, causal):
    q, k, v = inputs.dense_qkv(B, H, Nq, Nk, 128, seed=Nq + Nk)
    (q8, dq), (k8, dk), (v8, dv) = _quant(q, k, v)
    scale = default_scale(128)
    o, lse = _run(q8, k8, v8, (dq, dk, dv), causal, scale)
    o_ref, l_ref = oracle.attention(q8, k8, v8, scale, causal=causal, descales=(dq, dk, dv))
    compare("fp8_%dx%dx%dx%d_c%d" % (B, H, Nq, Nk, causal), o, lse, o_ref, l_ref, TOL_O_FP8, TOL_LSE)


@pytest.mark.parametrize("B,H,Nq,Nk,causal", [(1, 2, 300, 6200, False), (1, 1, 12300, 12300, True),
                                              (1, 1, 1000, 13000, True)])
def test_fp8_long_rows(B, H, Nq, Nk, causal):
    """Long rows (the decoupled prefill kernel): ragged tails, causal, Nq < Nk."""
    q, k, v = inputs.dense_qkv(B, H, Nq, Nk, 128, seed=Nq + Nk + 1)
    (q8, dq), (k8, dk), (v8, dv) = _quant(q, k, v)
    scale = default_scale(128)
    o, lse = _run(q8, k8, v8, (dq, dk, dv), causal, scale)
    q64, k64, v64 = (x.to(torch.float64) * s for x, s in ((q8, dq), (k8, dk), (v8, dv)))
    o_ref, l_ref = oracle.attention(q64.numpy(), k64.numpy(), v64.numpy(), scale, causal=causal)
    compare("fp8_long_%dx%dx%dx%d_c%d" % (B, H, Nq, Nk, causal), o, lse, o_ref, l_ref, TOL_O_FP8, TOL_LSE)


def test_fp8_workload_full():
    """B=2, H=16, N=8192, d=128: every output element against the oracle on the
    dequantised inputs.  The inputs are dequantised here, exactly, to float64
    (an e4m3 code has 4 significant bits and the descale 24, so each product
    is exact in float64; torch's e4m3 widening equals the oracle's decoder on
    every code, which the oracle pins check), and the oracle runs on those --
    the same numbers its own e4m3 path would form, without decoding every
    element once per row."""
    B, H, N, d = 2, 16, 8192, 128
    q, k, v = inputs.dense_qkv(B, H, N, N, d, seed=0)
    (q8, dq), (k8, dk), (v8, dv) = _quant(q, k, v)
    scale = default_scale(d)
    o, lse = _run(q8, k8, v8, (dq, dk, dv), False, scale)
    q64, k64, v64 = (x.to(torch.float64) * s for x, s in ((q8, dq), (k8, dk), (v8, dv)))
    o_ref, l_ref = oracle.attention(q64.numpy(), k64.numpy(), v64.numpy(), scale)
    compare("fp8_workload_full", o, lse, o_ref, l_ref, TOL_O_FP8, TOL_LSE)

