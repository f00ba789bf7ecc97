"""ctypes front end of the float64 attention oracle (test infrastructure only).

Compiles ``oracle.c`` with gcc on first use (or when ``build()`` is called)
into ``liboracle.so`` beside it, and converts arrays to the element codes the
C side decodes: float64, float32, bfloat16 bit patterns, e4m3fn bit patterns.
"""
import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

OR_F64, OR_F32, OR_BF16, OR_E4M3 = 0, 1, 2, 3
_ERRORS = {1: "invalid argument", 2: "out of host memory", 3: "sequence length or page id out of range"}


class OracleError(RuntimeError):
    pass


def build(force=False):
    """Compile oracle.c into liboracle.so (plain C, -O2, pthreads)."""
    global _lib
    with _lock:
        stale = (not os.path.exists(_LIB)) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)
        if force or stale:
            tmp = _LIB + ".%d.tmp" % os.getpid()
            cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", _SRC, "-o", tmp, "-lm"]
            subprocess.run(cmd, check=True)
            os.replace(tmp, _LIB)
            _lib = None
        if _lib is None:
            lib = ctypes.CDLL(_LIB)
            vp, i, i64, dbl = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double
            lib.oracle_attention.restype = i
            lib.oracle_attention.argtypes = [vp, i, dbl, vp, i, dbl, vp, i, dbl,
                                             i64, i64, i64, i, dbl, i, vp, i64, vp, vp, vp, i]
            lib.oracle_paged_decode.restype = i
            lib.oracle_paged_decode.argtypes = [vp, i, vp, vp, i, vp, vp, i, i, i, i, i, i64,
                                                dbl, vp, vp, vp, i]
            lib.oracle_paged_attention.restype = i
            lib.oracle_paged_attention.argtypes = [vp, i, vp, vp, i, vp, vp, vp, i, i64, i, i, i, i, i, i64,
                                                   dbl, i, vp, vp, vp, i]
            lib.oracle_attention_bwd.restype = i
            lib.oracle_attention_bwd.argtypes = [vp, vp, vp, vp, i, i64, i64, i64, i, dbl, i, vp, vp, vp, i]
            lib.oracle_decode.restype = i
            lib.oracle_decode.argtypes = [vp, i, i64, vp]
            _lib = lib
        return _lib


def default_threads():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def _as_raw(x):
    """Return (numpy array holding the raw elements, element code)."""
    try:
        import torch
    except ImportError:  # pragma: no cover
        torch = None
    if torch is not None and isinstance(x, torch.Tensor):
        if x.device.type != "cpu":
            raise OracleError("the oracle takes host (CPU) tensors only")
        x = x.contiguous()
        if x.dtype == torch.bfloat16:
            return x.view(torch.int16).numpy(), OR_BF16
        if x.dtype == torch.float8_e4m3fn:
            return x.view(torch.uint8).numpy(), OR_E4M3
        if x.dtype == torch.float32:
            return x.numpy(), OR_F32
        if x.dtype == torch.float64:
            return x.numpy(), OR_F64
        raise OracleError("unsupported tensor dtype %s" % x.dtype)
    a = np.ascontiguousarray(x)
    if a.dtype == np.float64:
        return a, OR_F64
    if a.dtype == np.float32:
        return a, OR_F32
    raise OracleError("unsupported array dtype %s" % a.dtype)


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def _check(rc):
    if rc != 0:
        raise OracleError("oracle failed: %s" % _ERRORS.get(rc, rc))


def attention(q, k, v, scale, causal=False, rows=None, descales=(1.0, 1.0, 1.0), nthreads=None,
              with_psum=False):
    """Exact attention for BHSD tensors q [B,H,Nq,d] (or [BH,Nq,d]), k, v [.., Nk, d].

    rows: optional int array of flattened row ids (bh * Nq + i).  Returns
    (o, lse) as float64 arrays, o shaped like q (or [len(rows), d]), lse like
    q without its last axis (or [len(rows)]); with_psum adds the per-row sum
    of probabilities computed in the third pass.
    """
    lib = build()
    qa, qd = _as_raw(q)
    ka, kd = _as_raw(k)
    va, vd = _as_raw(v)
    if qa.ndim < 2 or ka.shape[:-2] != qa.shape[:-2] or va.shape != ka.shape or ka.shape[-1] != qa.shape[-1]:
        raise OracleError("shape mismatch q%s k%s v%s" % (qa.shape, ka.shape, va.shape))
    lead = qa.shape[:-2]
    Nq, d = qa.shape[-2], qa.shape[-1]
    Nk = ka.shape[-2]
    BH = int(np.prod(lead)) if lead else 1
    if rows is None:
        n_rows, rptr = BH * Nq, None
        out_shape = tuple(lead) + (Nq,)
    else:
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        n_rows, rptr = rows.size, _ptr(rows)
        out_shape = (n_rows,)
    o = np.empty((n_rows, d), dtype=np.float64)
    lse = np.empty((n_rows,), dtype=np.float64)
    psum = np.empty((n_rows,), dtype=np.float64) if with_psum else None
    rc = lib.oracle_attention(_ptr(qa), qd, float(descales[0]), _ptr(ka), kd, float(descales[1]),
                              _ptr(va), vd, float(descales[2]), BH, Nq, Nk, d, float(scale),
                              int(bool(causal)), rptr, n_rows, _ptr(o), _ptr(lse),
                              _ptr(psum) if with_psum else None,
                              int(nthreads or default_threads()))
    _check(rc)
    res = (o.reshape(out_shape + (d,)), lse.reshape(out_shape))
    return res + (psum.reshape(out_shape),) if with_psum else res


def paged_decode(q, k_cache, v_cache, block_table, seq_lens, scale, nthreads=None, with_psum=False):
    """One-token attention per request over a paged cache.

    q [B,H,d]; k_cache, v_cache [num_pages, page_size, H, d]; block_table
    [B, max_pages] int32; seq_lens [B] int32.  Returns (o [B,H,d], lse [B,H]).
    """
    lib = build()
    qa, qd = _as_raw(q)
    ka, kd = _as_raw(k_cache)
    va, vd = _as_raw(v_cache)
    if kd != vd or ka.shape != va.shape:
        raise OracleError("k_cache and v_cache must match in shape and type")
    bt = np.ascontiguousarray(_to_numpy(block_table), dtype=np.int32)
    sl = np.ascontiguousarray(_to_numpy(seq_lens), dtype=np.int32)
    B, H, d = qa.shape
    num_pages, page_size, Hc, dc = ka.shape
    if (Hc, dc) != (H, d) or bt.shape[0] != B or sl.shape != (B,):
        raise OracleError("shape mismatch")
    o = np.empty((B * H, d), dtype=np.float64)
    lse = np.empty((B * H,), dtype=np.float64)
    psum = np.empty((B * H,), dtype=np.float64) if with_psum else None
    rc = lib.oracle_paged_decode(_ptr(qa), qd, _ptr(ka), _ptr(va), kd, _ptr(bt), _ptr(sl),
                                 B, H, d, page_size, bt.shape[1], num_pages, float(scale),
                                 _ptr(o), _ptr(lse), _ptr(psum) if with_psum else None,
                                 int(nthreads or default_threads()))
    _check(rc)
    res = (o.reshape(B, H, d), lse.reshape(B, H))
    return res + (psum.reshape(B, H),) if with_psum else res


def attention_bwd(q, k, v, dout, scale, causal=False, nthreads=None):
    """Gradients (dq, dk, dv) of attention(q, k, v) for the upstream gradient
    dout, all BHSD: q, dout [.., Nq, d], k, v [.., Nk, d] of one element type.
    Returned as float64 arrays shaped like q, k, v."""
    lib = build()
    qa, qd = _as_raw(q)
    ka, kd = _as_raw(k)
    va, vd = _as_raw(v)
    ga, gd = _as_raw(dout)
    if len({qd, kd, vd, gd}) != 1:
        raise OracleError("q, k, v and dout must share one element type")
    if ga.shape != qa.shape or va.shape != ka.shape or ka.shape[:-2] != qa.shape[:-2] or ka.shape[-1] != qa.shape[-1]:
        raise OracleError("shape mismatch")
    lead = qa.shape[:-2]
    Nq, d = qa.shape[-2], qa.shape[-1]
    Nk = ka.shape[-2]
    BH = int(np.prod(lead)) if lead else 1
    dq = np.empty(qa.shape, dtype=np.float64)
    dk = np.empty(ka.shape, dtype=np.float64)
    dv = np.empty(ka.shape, dtype=np.float64)
    _check(lib.oracle_attention_bwd(_ptr(qa), _ptr(ka), _ptr(va), _ptr(ga), qd, BH, Nq, Nk, d, float(scale),
                                    int(bool(causal)), _ptr(dq), _ptr(dk), _ptr(dv),
                                    int(nthreads or default_threads())))
    return dq, dk, dv


def paged_attention(q, k_cache, v_cache, block_table, seq_lens, scale, cu_seqlens_q=None, causal=False,
                    nthreads=None, with_psum=False):
    """Attention over a paged cache with grouped KV heads and several query
    tokens per request.

    q [total_q, H, d] token-major; k_cache, v_cache [num_pages, page_size,
    H_kv, d] with H % H_kv == 0 (query head h reads KV head h // (H // H_kv));
    block_table [B, max_pages] int32; seq_lens [B] int32 (keys per request,
    the new tokens' keys last); cu_seqlens_q [B+1] int32 token offsets, or
    None for one query token per request.  causal: query i of request r sees
    keys t <= seq_lens[r] - q_len_r + i.  Returns (o [total_q,H,d],
    lse [total_q,H]).
    """
    lib = build()
    qa, qd = _as_raw(q)
    ka, kd = _as_raw(k_cache)
    va, vd = _as_raw(v_cache)
    if kd != vd or ka.shape != va.shape:
        raise OracleError("k_cache and v_cache must match in shape and type")
    bt = np.ascontiguousarray(_to_numpy(block_table), dtype=np.int32)
    sl = np.ascontiguousarray(_to_numpy(seq_lens), dtype=np.int32)
    total_q, H, d = qa.shape
    num_pages, page_size, H_kv, dc = ka.shape
    B = sl.shape[0]
    if dc != d or bt.shape[0] != B or H % H_kv != 0:
        raise OracleError("shape mismatch")
    cu = None
    if cu_seqlens_q is not None:
        cu = np.ascontiguousarray(_to_numpy(cu_seqlens_q), dtype=np.int32)
        if cu.shape != (B + 1,):
            raise OracleError("cu_seqlens_q must have B + 1 entries")
    o = np.empty((total_q * H, d), dtype=np.float64)
    lse = np.empty((total_q * H,), dtype=np.float64)
    psum = np.empty((total_q * H,), dtype=np.float64) if with_psum else None
    rc = lib.oracle_paged_attention(_ptr(qa), qd, _ptr(ka), _ptr(va), kd, _ptr(bt),
                                    _ptr(cu) if cu is not None else None, _ptr(sl), B, total_q, H, H_kv, d,
                                    page_size, bt.shape[1], num_pages, float(scale), int(bool(causal)),
                                    _ptr(o), _ptr(lse), _ptr(psum) if with_psum else None,
                                    int(nthreads or default_threads()))
    _check(rc)
    res = (o.reshape(total_q, H, d), lse.reshape(total_q, H))
    return res + (psum.reshape(total_q, H),) if with_psum else res


def varlen_attention(q, k, v, cu_seqlens_q, cu_seqlens_k, scale, causal=False, nthreads=None):
    """Variable-length batch attention: request r owns query rows
    cu_seqlens_q[r] .. cu_seqlens_q[r+1]-1 of q [total_q, H, d] and key rows
    cu_seqlens_k[r] .. cu_seqlens_k[r+1]-1 of k, v [total_k, H_kv, d].

    The same computation as paged_attention on a cache of one-row pages
    (k viewed as [total_k, 1, H_kv, d]) whose table lists request r's rows in
    order; causal: query i sees keys t <= i + (k_len - q_len).  Returns
    (o [total_q, H, d], lse [total_q, H]).
    """
    import torch
    cu_q = torch.as_tensor(_to_numpy(cu_seqlens_q), dtype=torch.int32)
    cu_k = torch.as_tensor(_to_numpy(cu_seqlens_k), dtype=torch.int32)
    B = cu_k.shape[0] - 1
    lens = (cu_k[1:] - cu_k[:-1]).to(torch.int32)
    width = max(1, int(lens.max())) if B else 1
    table = torch.full((B, width), -1, dtype=torch.int32)
    for r in range(B):
        n = int(lens[r])
        table[r, :n] = torch.arange(int(cu_k[r]), int(cu_k[r]) + n, dtype=torch.int32)
    return paged_attention(q, k.unsqueeze(1), v.unsqueeze(1), table, lens, scale, cu_seqlens_q=cu_q,
                           causal=causal, nthreads=nthreads)


def decode_elems(x):
    """Widen every element of x (bf16 / e4m3fn / f32 / f64) to float64 via the C decoder."""
    lib = build()
    a, code = _as_raw(x)
    out = np.empty(a.size, dtype=np.float64)
    _check(lib.oracle_decode(_ptr(a), code, a.size, _ptr(out)))
    return out.reshape(a.shape)


def _to_numpy(x):
    try:
        import torch
        if isinstance(x, torch.Tensor):
            return x.detach().cpu().numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(x)
