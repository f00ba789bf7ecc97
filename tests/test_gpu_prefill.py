"""bf16 prefill parity: the CUDA path through the C ABI against the float64 oracle.

Covers the tiny (1x1x256x256, d=64), batched (4x16x2048x2048, d=128,
non-causal and causal) and long causal (1x32x32768x32768, d=128) workloads
in full -- the long one also on a stratified row sample, which fails fast --
and edge cases (on both prefill kernels -- the turn-based one for short rows,
the decoupled one for long rows):
ragged tails, a single row/key, Nq != Nk in both directions with the
bottom-right causal mask (including rows that see no key), large-magnitude
inputs, determinism, and guard bands around the outputs.
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
    attn.lib()  # fail loudly if the CUDA library is missing


def _run(q, k, v, causal, scale):
    o, lse = attn.fwd(q.to(DEV), k.to(DEV), v.to(DEV), causal=causal, scale=scale)
    attn.device_status()
    return o, lse


SMALL = [
    # B, H, Nq, Nk, d, causal
    (1, 1, 256, 256, 64, False),    # tiny workload
    (1, 1, 256, 256, 64, True),
    (1, 2, 300, 300, 128, True),    # ragged tail in both tiles
    (2, 1, 128, 384, 128, False),
    (1, 1, 1, 1, 64, False),        # one query, one key
    (1, 1, 1, 1, 128, True),
    (1, 3, 77, 77, 128, False),     # Nk < one KV block
    (1, 1, 5, 700, 128, True),      # Nq < Nk: bottom-right mask
    (1, 1, 700, 5, 128, True),      # Nq > Nk: leading rows see no key
    (1, 2, 257, 129, 64, False),
    (2, 2, 513, 1000, 64, True),
    (3, 2, 512, 512, 128, True),
    (1, 1, 640, 1111, 128, False),
]


@pytest.mark.parametrize("B,H,Nq,Nk,d,causal", SMALL)
def test_prefill_small(B, H, Nq, Nk, d, causal):
    q, k, v = inputs.dense_qkv(B, H, Nq, Nk, d, seed=B * 1000 + Nq + Nk + d)
    scale = default_scale(d)
    o, lse = _run(q, k, v, causal, scale)
    o_ref, l_ref = oracle.attention(q, k, v, scale, causal=causal)
    compare("prefill_%dx%dx%dx%d_d%d_c%d" % (B, H, Nq, Nk, d, causal), o, lse, o_ref, l_ref,
            TOL_O_BF16, TOL_LSE)


@pytest.mark.parametrize("causal", [False, True])
def test_prefill_batched_full(causal):
    """B=4, H=16, N=2048, d=128: every output element checked."""
    q, k, v = inputs.dense_qkv(4, 16, 2048, 2048, 128, seed=0)
    scale = default_scale(128)
    o, lse = _run(q, k, v, causal, scale)
    o_ref, l_ref = oracle.attention(q, k, v, scale, causal=causal)
    compare("prefill_batched_c%d" % causal, o, lse, o_ref, l_ref, TOL_O_BF16, TOL_LSE)


def test_prefill_long_causal_sampled():
    """B=1, H=32, N=32768, d=128, causal: every head on the stratified row set
    (first and last 128 rows, tile-boundary rows, 4096 random rows)."""
    B, H, N, d = 1, 32, 32768, 128
    q, k, v = inputs.dense_qkv(B, H, N, N, d, seed=0)
    scale = default_scale(d)
    o, lse = _run(q, k, v, True, scale)
    rows = inputs.sample_rows(B * H, N, n_random=4096, tile=128, seed=0)
    o_ref, l_ref = oracle.attention(q, k, v, scale, causal=True, rows=rows)
    ridx = torch.from_numpy(rows).to(DEV)
    compare("prefill_long_causal_sampled", o.reshape(-1, d).index_select(0, ridx),
            lse.reshape(-1).index_select(0, ridx), o_ref, l_ref, TOL_O_BF16, TOL_LSE)


# Long rows: a launch whose units stream 48 or more KV blocks on average runs
# on the decoupled kernel (S and P handed over separately); shorter ones on
# the turn-based kernel.  These shapes cover the decoupled kernel's edges.
LONG_ROWS = [
    # B, H, Nq, Nk, d, causal
    (1, 2, 300, 6200, 128, False),     # ragged tail in keys and queries
    (2, 1, 129, 6145, 128, False),     # one key past a whole block
    (1, 1, 700, 6300, 64, False),      # d = 64
    (1, 1, 12300, 12300, 128, True),   # causal, ragged last tile pair
    (1, 1, 1000, 13000, 128, True),    # Nq < Nk: bottom-right mask
    (1, 1, 13000, 12500, 128, True),   # Nq > Nk: the first 500 rows see no key
    (1, 1, 12544, 12544, 64, True),    # d = 64 causal
]


@pytest.mark.parametrize("B,H,Nq,Nk,d,causal", LONG_ROWS)
def test_prefill_long_rows(B, H, Nq, Nk, d, causal):
    q, k, v = inputs.dense_qkv(B, H, Nq, Nk, d, seed=B * 7000 + Nq + Nk + d)
    scale = default_scale(d)
    o, lse = _run(q, k, v, causal, scale)
    o_ref, l_ref = oracle.attention(q, k, v, scale, causal=causal)
    compare("prefill_long_%dx%dx%dx%d_d%d_c%d" % (B, H, Nq, Nk, d, causal), o, lse, o_ref, l_ref,
            TOL_O_BF16, TOL_LSE)


@pytest.mark.parametrize("mult", [4.0, 8.0])
def test_prefill_long_rows_large_magnitude(mult):
    """Long rows whose running max keeps rising: the O rescale of the decoupled kernel."""
    q, k, v = inputs.dense_qkv(1, 2, 256, 6200, 128, seed=15)
    q = (q.float() * mult).to(torch.bfloat16)
    k = (k.float() * mult).to(torch.bfloat16)
    scale = default_scale(128)
    o, lse = _run(q, k, v, False, scale)
    o_ref, l_ref = oracle.attention(q, k, v, scale)
    compare("prefill_long_mag%g" % mult, o, lse, o_ref, l_ref, TOL_O_BF16, TOL_LSE)
    # increasing scores along the keys: the max rises in block after block
    ramp = torch.linspace(0.0, 6.0, 6200).view(1, 1, 6200, 1)
    k2 = (k.float() + ramp * q.float().mean(dim=2, keepdim=True)).to(torch.bfloat16)
    o, lse = _run(q, k2, v, False, scale)
    o_ref, l_ref = oracle.attention(q, k2, v, scale)
    compare("prefill_long_ramp%g" % mult, o, lse, o_ref, l_ref, TOL_O_BF16, TOL_LSE)


def test_prefill_long_rows_guard_bands_and_no_lse():
    """Decoupled kernel: nothing outside O and LSE is written, results are
    deterministic, and a NULL LSE changes nothing else."""
    B, H, Nq, Nk, d = 1, 2, 333, 6300, 128
    q, k, v = (t.to(DEV) for t in inputs.dense_qkv(B, H, Nq, Nk, d, seed=16))
    n_o, n_l, g = B * H * Nq * d, B * H * Nq, 4096
    o_buf = torch.full((n_o + 2 * g,), 7.0, dtype=torch.bfloat16, device=DEV)
    l_buf = torch.full((n_l + 2 * g,), 7.0, dtype=torch.float32, device=DEV)
    o = o_buf[g:g + n_o].view(B, H, Nq, d)
    lse = l_buf[g:g + n_l].view(B, H, Nq)
    attn.fwd(q, k, v, causal=True, out=o, lse=lse)
    attn.device_status()
    for buf in (o_buf, l_buf):
        assert bool((buf[:g] == 7.0).all()) and bool((buf[-g:] == 7.0).all())
    o2, l2 = attn.fwd(q, k, v, causal=True)
    o3, _ = attn.fwd(q, k, v, causal=True, return_lse=False)
    attn.device_status()
    assert torch.equal(o, o2) and torch.equal(lse, l2) and torch.equal(o, o3)
    o_ref, l_ref = oracle.attention(q.cpu(), k.cpu(), v.cpu(), default_scale(d), causal=True)
    compare("prefill_long_guard", o, lse, o_ref, l_ref, TOL_O_BF16, TOL_LSE)


def test_prefill_long_causal_full():
    """B=1, H=32, N=32768, d=128, causal: every output element of the
    1,048,576 rows (about 8.8 TFLOP of float64 oracle work)."""
    B, H, N, d = 1, 32, 32768, 128
    q, k, v = inputs.dense_qkv(B, H, N, N, d, seed=0)
    scale = default_scale(d)
    o, lse = _run(q, k, v, True, scale)
    o_ref, l_ref = oracle.attention(q, k, v, scale, causal=True)
    compare("prefill_long_causal_full", o, lse, o_ref, l_ref, TOL_O_BF16, TOL_LSE)


@pytest.mark.parametrize("mult", [4.0, 8.0])
def test_prefill_large_magnitude(mult):
    """Scores with a spread of hundreds: exp without max subtraction would
    overflow; the running-max update must keep everything finite."""
    q, k, v = inputs.dense_qkv(1, 2, 384, 384, 128, seed=5)
    q = (q.float() * mult).to(torch.bfloat16)
    k = (k.float() * mult).to(torch.bfloat16)
    scale = default_scale(128)
    for causal in (False, True):
        o, lse = _run(q, k, v, causal, scale)
        o_ref, l_ref = oracle.attention(q, k, v, scale, causal=causal)
        compare("prefill_mag%g_c%d" % (mult, causal), o, lse, o_ref, l_ref, TOL_O_BF16, TOL_LSE)


def test_prefill_deterministic_and_no_lse():
    q, k, v = (t.to(DEV) for t in inputs.dense_qkv(2, 4, 1000, 1000, 128, seed=11))
    o1, l1 = attn.fwd(q, k, v, causal=True)
    o2, l2 = attn.fwd(q, k, v, causal=True)
    o3, _ = attn.fwd(q, k, v, causal=True, return_lse=False)
    attn.device_status()
    assert torch.equal(o1, o2) and torch.equal(l1, l2) and torch.equal(o1, o3)


def test_prefill_guard_bands():
    """Nothing outside O [B,H,Nq,d] and LSE [B,H,Nq] is written."""
    B, H, Nq, Nk, d = 1, 3, 333, 257, 128
    q, k, v = (t.to(DEV) for t in inputs.dense_qkv(B, H, Nq, Nk, d, seed=12))
    n_o, n_l, g = B * H * Nq * d, B * H * Nq, 4096
    o_buf = torch.full((n_o + 2 * g,), 7.0, dtype=torch.bfloat16, device=DEV)
    l_buf = torch.full((n_l + 2 * g,), 7.0, dtype=torch.float32, device=DEV)
    o = o_buf[g:g + n_o].view(B, H, Nq, d)
    lse = l_buf[g:g + n_l].view(B, H, Nq)
    attn.fwd(q, k, v, causal=True, out=o, lse=lse)
    attn.device_status()
    for buf in (o_buf, l_buf):
        assert bool((buf[:g] == 7.0).all()) and bool((buf[-g:] == 7.0).all())
    o_ref, l_ref = oracle.attention(q.cpu(), k.cpu(), v.cpu(), default_scale(d), causal=True)
    compare("prefill_guard", o, lse, o_ref, l_ref, TOL_O_BF16, TOL_LSE)


def test_prefill_scale_is_honoured():
    q, k, v = inputs.dense_qkv(1, 1, 200, 300, 64, seed=13)
    for scale in (0.01, 0.5):
        o, lse = _run(q, k, v, False, scale)
        o_ref, l_ref = oracle.attention(q, k, v, float(np.float32(scale)))
        compare("prefill_scale%g" % scale, o, lse, o_ref, l_ref, TOL_O_BF16, TOL_LSE)
