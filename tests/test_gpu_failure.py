"""Failure handling without a GPU fault.

Every wait in the library's kernels is bounded: after the limit the kernel
records ATTN_ERR_TIMEOUT in the device status word and returns.  The
self-test kernel waits, through that same bounded wait, on a barrier that
nothing completes.  The host must then read ATTN_ERR_TIMEOUT; attention
launches enqueued while the word is set must leave their outputs untouched;
and once the word is read (and cleared) the context must compute correctly.
Nothing here traps, faults or hangs the GPU: the wait gives up by itself.
"""
import pytest
import torch

import attention_attn_fwd_03_gb300 as attn
import oracle
from attention_attn_fwd_03_gb300 import inputs

from _parity import TOL_LSE, TOL_O_BF16, compare, default_scale

pytestmark = pytest.mark.gpu
DEV = "cuda"


def test_bounded_wait_reports_timeout_and_the_context_survives():
    attn.lib()
    q, k, v = inputs.dense_qkv(1, 2, 300, 300, 128, seed=8)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    sentinel = torch.full((1, 2, 300, 128), 3.0, dtype=torch.bfloat16, device=DEV)
    out = sentinel.clone()
    lse = torch.full((1, 2, 300), 7.0, dtype=torch.float32, device=DEV)
    stream = torch.cuda.current_stream().cuda_stream
    assert attn.attn_selftest_wait_timeout(stream) == attn.ATTN_OK
    attn.fwd(qd, kd, vd, causal=True, out=out, lse=lse)  # runs after the wait gave up: must do nothing
    with pytest.raises(attn.AttnError) as ei:
        attn.device_status()
    assert ei.value.status == attn.ATTN_ERR_TIMEOUT
    assert torch.equal(out, sentinel) and bool((lse == 7.0).all())
    attn.device_status()  # the word was cleared by the read above
    scale = default_scale(128)
    o, l = attn.fwd(qd, kd, vd, causal=True, scale=scale)
    attn.device_status()
    o_ref, l_ref = oracle.attention(q, k, v, scale, causal=True)
    compare("after_timeout", o, l, o_ref, l_ref, TOL_O_BF16, TOL_LSE)
