"""Host-staged prefill (attn_fwd_host): inputs and outputs in host memory, the
(b, h) range pipelined in chunks through copy-in, kernels and copy-out.

Each (b, h) problem runs through the same kernel as attn_fwd, so the outputs
must equal attn_fwd on device copies bit for bit, for every chunk size
(one pair, ragged last chunk, the default, larger than B*H) and for several
mask modes in one call.  Also: parity with the float64 oracle, pageable host
buffers, a NULL LSE for one mode, ordering after work already on the stream,
repeated calls reusing the slots, and device pointers refused.
"""
import ctypes

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


def _pinned(t):
    return t.contiguous().pin_memory()


def _device_ref(q, k, v, causal, scale):
    o, lse = attn.fwd(q.to(DEV), k.to(DEV), v.to(DEV), causal=causal, scale=scale)
    attn.device_status()
    return o.cpu(), lse.cpu()


@pytest.mark.parametrize("B,H,Nq,Nk,d,chunk", [
    (2, 4, 300, 300, 128, 1),     # one pair per chunk, more chunks than slots
    (2, 4, 300, 300, 128, 3),     # ragged last chunk (3, 3, 2)
    (1, 8, 257, 640, 64, 0),      # default chunk
    (2, 2, 130, 77, 128, 100),    # chunk larger than B*H: one chunk
    (3, 5, 513, 513, 128, 4),
    (1, 3, 200, 6300, 128, 1),    # long rows: the decoupled prefill kernel, one head per chunk
])
def test_bit_identical_to_device_path(B, H, Nq, Nk, d, chunk):
    q, k, v = (_pinned(t) for t in inputs.dense_qkv(B, H, Nq, Nk, d, seed=B * 100 + H + Nq + chunk))
    scale = default_scale(d)
    outs, lses = attn.fwd_host(q, k, v, causal=(False, True), scale=scale, chunk_bh=chunk)
    attn.device_status()
    for m, causal in enumerate((False, True)):
        o_ref, l_ref = _device_ref(q, k, v, causal, scale)
        assert torch.equal(outs[m], o_ref), "mode %d: O differs from attn_fwd" % m
        assert torch.equal(lses[m], l_ref), "mode %d: LSE differs from attn_fwd" % m


def test_oracle_parity_and_null_lse():
    B, H, Nq, Nk, d = 2, 3, 384, 500, 128
    q, k, v = (_pinned(t) for t in inputs.dense_qkv(B, H, Nq, Nk, d, seed=77))
    scale = default_scale(d)
    lse1 = torch.empty((B, H, Nq), dtype=torch.float32).pin_memory()
    outs, lses = attn.fwd_host(q, k, v, causal=(True, False), scale=scale, chunk_bh=2, lse=[lse1, None])
    attn.device_status()
    assert lses[1] is None
    o_ref, l_ref = oracle.attention(q, k, v, scale, causal=True)
    compare("host_staged_causal", outs[0], lses[0], o_ref, l_ref, TOL_O_BF16, TOL_LSE)
    o_ref2, _ = _device_ref(q, k, v, False, scale)
    assert torch.equal(outs[1], o_ref2)


def test_pageable_buffers_give_the_same_result():
    B, H, N, d = 1, 6, 400, 128
    q, k, v = inputs.dense_qkv(B, H, N, N, d, seed=5)
    q, k, v = q.contiguous(), k.contiguous(), v.contiguous()
    assert not q.is_pinned()
    out = [torch.empty((B, H, N, d), dtype=torch.bfloat16)]
    lse = [torch.empty((B, H, N), dtype=torch.float32)]
    attn.fwd_host(q, k, v, causal=(True,), chunk_bh=4, out=out, lse=lse)
    attn.device_status()
    o_ref, l_ref = _device_ref(q, k, v, True, default_scale(d))
    assert torch.equal(out[0], o_ref) and torch.equal(lse[0], l_ref)


def test_copies_start_after_earlier_work_on_the_stream():
    """A device->host copy enqueued just before the call rewrites the host Q;
    the call must read the new values, and repeated calls reuse the slots."""
    B, H, N, d = 2, 4, 256, 128
    q0, k, v = (_pinned(t) for t in inputs.dense_qkv(B, H, N, N, d, seed=11))
    q1 = inputs.dense_qkv(B, H, N, N, d, seed=12)[0].to(DEV)
    hq = q0.clone().pin_memory()
    ws = torch.empty(attn.attn_fwd_host_workspace_size(B, H, N, N, d, 1, 2), dtype=torch.uint8, device=DEV)
    for it in range(3):
        hq.copy_(q0)
        torch.cuda.synchronize()
        hq.copy_(q1, non_blocking=True)  # on the current stream, not yet complete when the call enqueues
        outs, lses = attn.fwd_host(hq, k, v, causal=(False,), chunk_bh=2, workspace=ws)
        attn.device_status()
        o_ref, l_ref = _device_ref(q1.cpu(), k, v, False, default_scale(d))
        assert torch.equal(outs[0], o_ref) and torch.equal(lses[0], l_ref), "iteration %d" % it


def test_device_pointers_are_refused():
    B, H, N, d = 1, 2, 128, 128
    q, k, v = (t.to(DEV) for t in inputs.dense_qkv(B, H, N, N, d, seed=3))
    hq = q.cpu().pin_memory()
    ws_bytes = attn.attn_fwd_host_workspace_size(B, H, N, N, d, 1, 0)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=DEV)
    modes = (ctypes.c_int * 1)(0)
    host_out = torch.empty((B, H, N, d), dtype=torch.bfloat16).pin_memory()
    outs = (ctypes.c_void_p * 1)(host_out.data_ptr())
    st = attn.attn_fwd_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), 1, ctypes.addressof(modes),
                            ctypes.addressof(outs), None, B, H, N, N, d, 0.088, 0, ws.data_ptr(), ws_bytes, None)
    assert st == attn.ATTN_ERR_INVALID_ARG
    dev_out = torch.empty((B, H, N, d), dtype=torch.bfloat16, device=DEV)
    outs_dev = (ctypes.c_void_p * 1)(dev_out.data_ptr())
    hk, hv = k.cpu().pin_memory(), v.cpu().pin_memory()
    st = attn.attn_fwd_host(hq.data_ptr(), hk.data_ptr(), hv.data_ptr(), 1, ctypes.addressof(modes),
                            ctypes.addressof(outs_dev), None, B, H, N, N, d, 0.088, 0, ws.data_ptr(), ws_bytes,
                            None)
    assert st == attn.ATTN_ERR_INVALID_ARG
    st = attn.attn_fwd_host(hq.data_ptr(), hk.data_ptr(), hv.data_ptr(), 1, ctypes.addressof(modes),
                            ctypes.addressof(outs), None, B, H, N, N, d, 0.088, 0, host_out.data_ptr(), ws_bytes,
                            None)
    assert st == attn.ATTN_ERR_WORKSPACE  # host memory as workspace
    attn.device_status()
